"""Selection reuse across steps on the GPU (ice_select_attn_reuse) against the
oracle's ReuseOracle, step by step: the reuse decisions, the pages and the
attention, with inserted tokens between steps, for the device and host pools."""
import numpy as np
import pytest
import torch

from tests.parity_helpers import ATOL, oracle_for_unit, q_of_unit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from semantic_paged_kv_head_gb300 import build
    build.build_lib()
    from semantic_paged_kv_head_gb300 import ice as m
    return m


@pytest.mark.parametrize("kv_host", [False, True])
def test_reuse_follows_oracle(ice, kv_host):
    from oracle import oracle as O
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=3, n_tokens=800, n_insert=60,
                     n_centers=16, seed=23)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             max_tokens=w.n_tokens + w.n_insert, kv_host=kv_host)
    U, n_sel, r = w.n_units, w.budget // w.page_size, 2
    orcs = [O.ReuseOracle(oracle_for_unit(w, keys, values, u), r) for u in range(U)]
    page_ids = torch.full((U, n_sel), -1, dtype=torch.int32, device="cuda")
    n_pages = torch.zeros((U,), dtype=torch.int32, device="cuda")
    flags = torch.zeros((U,), dtype=torch.int32, device="cuda")
    # the query of each step: repeated queries (reuse), new ones (reselect)
    schedule = [0, 0, 0, 0, 1, 1, 2, 2, 2, 2, 2, 3]
    n_ins = 0
    seen_reuse = seen_select = 0
    for step, qi in enumerate(schedule):
        if step == 5:  # tokens generated between steps, into every unit
            for _ in range(30):
                k, v = synth.make_insert_token(w, centers, deltas, n_ins)
                gix.insert(k.cuda(), v.cuda())
                for u in range(U):
                    orcs[u].ix.insert(k.view(-1, w.d)[u], v.view(-1, w.d)[u])
                n_ins += 1
        q = synth.make_queries(w, centers, step=qi, drift_deltas=deltas)
        out, _, _ = gix.select_attn_reuse(q.cuda(), w.budget, r, page_ids, n_pages, reselected=flags)
        torch.cuda.synchronize()
        assert gix.get_error() == 0
        for u in range(U):
            ids_o, npg_o, resel_o, out_o = orcs[u].step(q_of_unit(w, q, u), w.budget)
            assert int(flags[u]) == int(resel_o), (step, u)
            assert int(n_pages[u]) == npg_o, (step, u)
            assert np.array_equal(page_ids[u, :npg_o].cpu().numpy(), ids_o[:npg_o]), (step, u)
            got = out.view(-1, w.group, w.d)[u].float().cpu().numpy()
            assert np.max(np.abs(got - out_o)) <= ATOL[w.dtype], (step, u)
            seen_reuse += not resel_o
            seen_select += resel_o
    assert seen_reuse > 0 and seen_select > 0
    # reset: every unit selects again
    gix.reuse_reset()
    q = synth.make_queries(w, centers, step=3, drift_deltas=deltas)
    gix.select_attn_reuse(q.cuda(), w.budget, r, page_ids, n_pages, reselected=flags)
    torch.cuda.synchronize()
    assert int(flags.sum()) == U


def test_reuse_r0_equals_select_attn(ice):
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2, n_tokens=1500,
                     n_centers=16, seed=29)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers).cuda()
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed)
    U, n_sel = w.n_units, w.budget // w.page_size
    out_a, ids_a, npg_a = gix.select_attn(q, w.budget)
    ids = torch.full((U, n_sel), -1, dtype=torch.int32, device="cuda")
    npg = torch.zeros((U,), dtype=torch.int32, device="cuda")
    for _ in range(3):
        out_b, _, _ = gix.select_attn_reuse(q, w.budget, 0, ids, npg)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_a) and torch.equal(npg, npg_a)
        assert torch.equal(out_b, out_a)
    assert gix.get_error() == 0

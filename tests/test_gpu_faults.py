"""Failure paths on the GPU without a GPU fault: host-side argument errors on a
live index, device-side bounds and capacity reports, and the fused call's
bounded wait forced to run out by a test flag (ICE_ERR_TIMEOUT; the context
stays usable)."""
import ctypes

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


@pytest.fixture(scope="module")
def small(ice):
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=2, n_tokens=900,
                     n_centers=8, seed=31)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers).cuda()
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed)
    return w, gix, q


def test_host_argument_errors_on_a_live_index(ice, small):
    w, gix, q = small
    raw = ice.raw_library()
    U, n_sel = gix.n_units, w.budget // w.page_size
    ids = torch.zeros((U, n_sel), dtype=torch.int32, device="cuda")
    npg = torch.zeros((U,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    h, s = gix._h, torch.cuda.current_stream().cuda_stream
    qp, ip, np_, op = q.data_ptr(), ids.data_ptr(), npg.data_ptr(), out.data_ptr()
    E = ice.ICE_ERR_INVALID_ARG
    assert raw.ice_select(h, None, w.budget, ip, np_, None, s) == E
    assert raw.ice_select(h, qp + 2, w.budget, ip, np_, None, s) == E  # misaligned
    assert raw.ice_select(h, qp, w.page_size - 1, ip, np_, None, s) == E  # budget < P
    assert raw.ice_select(h, qp, w.budget + 1, ip, np_, None, s) == E  # not a multiple of P
    assert raw.ice_select(h, qp, w.budget, None, np_, None, s) == E
    assert raw.ice_select_attn(h, qp, w.budget, ip, np_, None, None, s) == E
    assert raw.ice_select_attn(h, qp, w.budget, ip, np_, None, op + 4, s) == E
    assert raw.ice_sparse_attn(h, qp, ip, np_, 0, op, s) == E  # page_stride 0
    assert raw.ice_sparse_attn(h, qp, ip, None, n_sel, op, s) == E
    assert raw.ice_select_attn_reuse(h, qp, w.budget, -1, ip, np_, None, op, s) == E  # r < 0
    assert raw.ice_insert(h, None, None, s) == E
    assert raw.ice_debug_set_flags(h, 1 << 5) == E
    assert raw.ice_select(None, qp, w.budget, ip, np_, None, s) == E
    # nothing was launched: the index still answers normally
    gix.select(q, w.budget, ids, npg)
    torch.cuda.synchronize()
    assert gix.get_error() == 0


def test_forced_timeout_reports_and_recovers(ice, small):
    w, gix, q = small
    ref, ids_ref, npg_ref = gix.select_attn(q, w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    gix.debug_set_flags(ice.DEBUG_STALL_ATTN)
    out, ids, npg = gix.select_attn(q, w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == ice.ICE_ERR_TIMEOUT
    assert torch.equal(ids, ids_ref) and torch.equal(npg, npg_ref)  # the selection is unaffected
    assert float(out.float().abs().max()) == 0.0  # the attention of the stalled round is skipped
    gix.debug_set_flags(0)
    out2, _, _ = gix.select_attn(q, w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    assert torch.equal(out2, ref)


def test_forced_timeout_over_several_staging_rounds(ice):
    """A selection larger than the fused kernel's staging region (64 pages of
    up to 16 fp32 rows each) is attended in several rounds; a forced timeout in
    the first round ends the attention there: no further copies are issued on
    the barrier, the status reports the timeout, the output is zero and the
    next call on the same index is exact."""
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["tiny_fp32_4k"], n_tokens=4096, n_centers=16, seed=33,
                     budget=1024)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers).cuda()
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed)
    ref, ids_ref, npg_ref = gix.select_attn(q, w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    d = gix.dump(0)
    rows = sum(int(d["comp"][0]["list_cnt"][p]) for p in ids_ref[0, :int(npg_ref[0])].tolist())
    assert rows * 2 * 128 * 4 > 100 * 1024  # more K and V rows than one staging round holds
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


def test_insert_capacity_is_reported(ice):
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["mistral7b_gen8k"], n_kv_heads=1, n_tokens=40, n_insert=3,
                     n_centers=4, seed=37)
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    gix = ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                             n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                             max_tokens=w.n_tokens + 2)
    for s in range(2):
        k, v = synth.make_insert_token(w, centers, deltas, s)
        gix.insert(k.cuda(), v.cuda())
    k, v = synth.make_insert_token(w, centers, deltas, 2)
    with pytest.raises(ice.IceError) as ei:
        gix.insert(k.cuda(), v.cuda())
    assert ei.value.code == ice.ICE_ERR_CAPACITY
    torch.cuda.synchronize()
    assert gix.get_error() == 0

"""Decode-step calls on page-locked host buffers: the kernels read q, k, v and
write out, page ids and counts in place over the CPU-GPU link. Results equal
those of the same calls on device buffers bit for bit, and memory the GPU
cannot address is refused before anything is launched."""
import ctypes

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


def _workload(dtype=torch.bfloat16):
    from semantic_paged_kv_head_gb300 import synth
    return synth, synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2,
                               n_tokens=1500, n_insert=6, n_centers=24, dtype=dtype, seed=71)


def _build(ice, w, keys, values):
    return ice.IceIndex.build(keys.cuda(), values.cuda(), page_size=w.page_size,
                              n_q_heads=w.n_q_heads, n_composite=w.n_composite, seed=w.seed,
                              max_tokens=w.n_tokens + w.n_insert)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_select_attn_on_host_buffers(ice, dtype):
    synth, w = _workload(dtype)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    gix = _build(ice, w, keys, values)
    out_d, ids_d, n_d = gix.select_attn(q.cuda(), w.budget)
    q_h = q.pin_memory()
    out_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    U, n_sel = w.n_units, w.budget // w.page_size
    ids_h = torch.empty((U, n_sel), dtype=torch.int32).pin_memory()
    n_h = torch.empty((U,), dtype=torch.int32).pin_memory()
    gix.select_attn(q_h, w.budget, out_h, ids_h, n_h)
    torch.cuda.synchronize()
    assert gix.get_error() == 0
    assert torch.equal(ids_h, ids_d.cpu()) and torch.equal(n_h, n_d.cpu())
    assert torch.equal(out_h, out_d.cpu())
    # and the oracle agrees with what landed in host memory
    for u in (0, U - 1):
        orc = oracle_for_unit(w, keys, values, u)
        check_select_attn(w, orc, q_of_unit(w, q, u), ids_h[u], n_h[u],
                          out_h.view(-1, w.group, w.d)[u], None, f"unit {u}")
    # the separate calls on host buffers too
    ids2, n2 = gix.select(q_h, w.budget)
    out2 = gix.sparse_attn(q_h, ids_h, n_h)
    torch.cuda.synchronize()
    assert torch.equal(ids2.cpu(), ids_d.cpu()) and torch.equal(n2.cpu(), n_d.cpu())
    assert not out2.is_cuda and out2.is_pinned()


def test_decode_step_and_insert_on_host_buffers(ice):
    synth, w = _workload()
    keys, values, centers = synth.make_kv(w)
    deltas = synth.make_drift(w, centers)
    a, b = _build(ice, w, keys, values), _build(ice, w, keys, values)
    U, n_sel = w.n_units, w.budget // w.page_size
    ids_a = torch.empty((U, n_sel), dtype=torch.int32, device="cuda")
    n_a = torch.empty((U,), dtype=torch.int32, device="cuda")
    ids_b = torch.empty((U, n_sel), dtype=torch.int32).pin_memory()
    n_b = torch.empty((U,), dtype=torch.int32).pin_memory()
    for t in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, t)
        q = synth.make_queries(w, centers, step=t, drift_deltas=deltas)
        out_a = torch.empty_like(q.cuda())
        out_b = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        if t % 2 == 0:
            a.decode_step(k.cuda(), v.cuda(), q.cuda(), w.budget, ids_a, n_a, out_a)
            b.decode_step(k.pin_memory(), v.pin_memory(), q.pin_memory(), w.budget, ids_b, n_b, out_b)
        else:
            a.insert(k.cuda(), v.cuda())
            b.insert(k.pin_memory(), v.pin_memory())
            a.select_attn(q.cuda(), w.budget, out_a, ids_a, n_a)
            b.select_attn(q.pin_memory(), w.budget, out_b, ids_b, n_b)
        torch.cuda.synchronize()
        assert torch.equal(ids_b, ids_a.cpu()) and torch.equal(n_b, n_a.cpu()), t
        assert torch.equal(out_b, out_a.cpu()), t
    for u in range(U):
        da, db = a.dump(u), b.dump(u)
        assert da["n"] == db["n"]
        for l in range(len(da["comp"])):
            assert (da["comp"][l]["slot_tok"] == db["comp"][l]["slot_tok"]).all()
    assert a.get_error() == 0 and b.get_error() == 0


def test_unaddressable_memory_is_refused(ice):
    """Pageable host memory given straight to the C ABI: refused on the host
    (nothing launched), and the index keeps working."""
    synth, w = _workload()
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    gix = _build(ice, w, keys, values)
    U, n_sel = w.n_units, w.budget // w.page_size
    q_pageable = q.clone()  # ordinary CPU memory
    assert not q_pageable.is_pinned()
    ids = torch.empty((U, n_sel), dtype=torch.int32, device="cuda")
    n = torch.empty((U,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q.cuda())
    lib = ice._lib
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    r = lib.ice_select_attn(gix._h, ctypes.c_void_p(q_pageable.data_ptr()), w.budget,
                            ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(n.data_ptr()), None,
                            ctypes.c_void_p(out.data_ptr()), st)
    assert r == ice.ICE_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        gix.select_attn(q_pageable, w.budget)
    out2, ids2, n2 = gix.select_attn(q.cuda(), w.budget)
    torch.cuda.synchronize()
    assert gix.get_error() == 0 and int(n2.min()) > 0

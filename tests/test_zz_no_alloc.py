"""The allocation-free key-code call against the build's own codes.

ice_key_codes_noalloc serves callers that cannot allocate device memory while
they run. It computes the same per-token Morton keys and per-unit scale
exponents that ice_build indexes, with its scratch in fixed device arrays of the
library. This test compares the two, on two calls in a row with different
inputs (the shared scratch must be reset between calls), through the C ABI.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _codes_from_build(ice, gix, U, n, L):
    """Morton key of every token and e of every unit, read from the index."""
    mk = np.zeros((L, U, n), dtype=np.uint64)
    e = np.zeros(U, dtype=np.int64)
    for u in range(U):
        d = gix.dump(u)
        e[u] = d["e"]
        for l, comp in enumerate(d["comp"]):
            for i in range(d["n_leaf"][l]):
                lid, c = int(comp["id"][i]), int(comp["cnt"][i])
                toks = comp["slot_tok"][lid, :c]
                mk[l, u, toks] = comp["slot_key"][lid, :c]
    return mk, e


def test_noalloc_key_codes_match_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from semantic_paged_kv_head_gb300 import build
    build.build_lib()
    from semantic_paged_kv_head_gb300 import ice, synth

    cases = [
        synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=2, n_kv_heads=2, n_tokens=3001,
                     n_centers=32, seed=21),
        synth.scaled(synth.WORKLOADS["tiny_fp32_4k"], n_tokens=2500, n_centers=16, seed=22,
                     n_composite=2),
    ]
    for w in cases:  # two calls in a row, different shapes, dtypes and norms
        keys, values, _ = synth.make_kv(w)
        if w.dtype == torch.float32:
            keys = keys * 3.0  # a different scale exponent than the first call
        kd, vd = keys.cuda(), values.cuda()
        U, n, L = w.n_units, w.n_tokens, w.n_composite
        gix = ice.IceIndex.build(kd, vd, page_size=w.page_size, n_q_heads=w.n_q_heads,
                                 n_composite=L, seed=w.seed)
        ref_mk, ref_e = _codes_from_build(ice, gix, U, n, L)
        mk, e = ice.key_codes_noalloc(kd, n_composite=L, seed=w.seed)
        torch.cuda.synchronize()
        assert np.array_equal(e.cpu().numpy().astype(np.int64), ref_e)
        assert np.array_equal(mk.cpu().numpy().view(np.uint64), ref_mk)


def test_noalloc_rejects_oversize():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from semantic_paged_kv_head_gb300 import ice
    keys = torch.zeros((1, 1, 1, (1 << 20) + 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ice.IceError) as ei:
        ice.key_codes_noalloc(keys)
    assert ei.value.code == ice.ICE_ERR_CAPACITY

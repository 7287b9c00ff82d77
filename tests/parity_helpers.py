"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and the oracle on the same seeded inputs, and compare.

Tolerances (attention output, max-abs): 2e-2 for bf16 inputs/outputs, 1e-5
for fp32. Page ids, leaf tables, codes and token placement must match exactly.
"""
import numpy as np
import torch

ATOL = {torch.bfloat16: 2e-2, torch.float32: 1e-5}


def unit_slices(w, u):
    """(b, layer, kv_head) of unit u."""
    h = u % w.n_kv_heads
    r = u // w.n_kv_heads
    return r // w.n_layers, r % w.n_layers, h


def oracle_for_unit(w, keys, values, u, forced_e=None):
    from oracle.oracle import OracleIndex
    b, ly, h = unit_slices(w, u)
    ix = OracleIndex(w.d, w.n_proj, w.n_composite, w.page_size, w.seed, w.dir_kind)
    ix.build(keys[b, ly, h].cpu(), values[b, ly, h].cpu(), forced_e=forced_e)
    return ix


def q_of_unit(w, q, u):
    b, ly, h = unit_slices(w, u)
    G = w.group
    return q[b, ly, h * G:(h + 1) * G].cpu()


def compare_index(gdump, orc, unit_label=""):
    """GPU leaf tables / lists of one unit == oracle canonical dump (exact)."""
    assert gdump["e"] == orc.e, unit_label
    assert gdump["n"] == orc.n, unit_label
    P = gdump["P"]
    tok_loc = gdump["tok_loc"]
    for l, comp in enumerate(gdump["comp"]):
        od = orc.dump(l)
        N = gdump["n_leaf"][l]
        assert N == len(od["t"]), (unit_label, l, N, len(od["t"]))
        assert gdump["next_id"][l] == orc.next_id(l), (unit_label, l)
        assert np.array_equal(comp["t"][:N], od["t"]), (unit_label, l)
        assert np.array_equal(comp["rec_t"][:N], od["t"]), (unit_label, l)
        assert np.array_equal(comp["pm"][:N], od["pm"]), (unit_label, l)
        assert np.array_equal(comp["pt"][:N], od["pt"]), (unit_label, l)
        assert np.array_equal(comp["id"][:N], od["id"]), (unit_label, l)
        assert np.array_equal(comp["cnt"][:N], od["cnt"]), (unit_label, l)
        assert np.array_equal(comp["lo"][:N], od["lo"]), (unit_label, l)
        assert np.array_equal(comp["hi"][:N], od["hi"]), (unit_label, l)
        mk, _ = orc.token_keys(l)
        for i in range(N):
            lid, c = int(comp["id"][i]), int(comp["cnt"][i])
            assert comp["list_cnt"][lid] == c
            toks = comp["slot_tok"][lid, :c]
            assert np.array_equal(np.sort(toks), od["toks"][od["off"][i]:od["off"][i + 1]]), (
                unit_label, l, i)
            assert np.array_equal(comp["slot_key"][lid, :c], mk[toks]), (unit_label, l, i)
            if l == 0:
                assert np.array_equal(tok_loc[toks], lid * P + np.arange(c)), (unit_label, i)
            if l == 1:  # composite-1 slots carry their token's page row, both ways
                assert np.array_equal(gdump["slot_loc1"][lid, :c], tok_loc[toks]), (unit_label, i)
                assert np.array_equal(gdump["tok_slot1"][toks], lid * P + np.arange(c)), (unit_label, i)


def compare_pages(gix, w, keys, values, gdump, u, max_pages=8):
    """Page rows hold exactly the K/V rows of the slot tokens."""
    b, ly, h = unit_slices(w, u)
    K = keys[b, ly, h].cpu()
    V = values[b, ly, h].cpu()
    comp = gdump["comp"][0]
    N = gdump["n_leaf"][0]
    for i in list(range(min(N, max_pages // 2))) + list(range(max(0, N - max_pages // 2), N)):
        lid, c = int(comp["id"][i]), int(comp["cnt"][i])
        hk, hv = gix.page(u, lid)
        toks = torch.from_numpy(comp["slot_tok"][lid, :c].astype(np.int64))
        assert torch.equal(hk[:c], K[toks]) and torch.equal(hv[:c], V[toks]), (u, i)


def check_select_attn(w, orc, q_u, gids, gnp, gout, gstats=None, label=""):
    """Page ids bit-exact, attention within tolerance, stats == oracle trace."""
    ids, npg, tr = orc.select(q_u, w.budget)
    n_sel = w.budget // w.page_size
    assert int(gnp) == npg, (label, int(gnp), npg)
    assert np.array_equal(gids.cpu().numpy()[:n_sel], ids), (label, gids.cpu().numpy(), ids)
    ref = orc.attn(q_u, ids, npg)
    got = gout.float().cpu().numpy().astype(np.float64)
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= ATOL[w.dtype], (label, err)
    if gstats is not None:
        s = gstats.cpu().numpy()
        assert s[0] == tr["leaves"] and s[1] == tr["cands"] and s[2] == tr["sel_tokens"], (label, s, tr)
    return err, tr

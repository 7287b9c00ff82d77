"""Where the selection's recall goes (CPU, oracle only).

recall@k (k = the token budget) compares the tokens of the selected pages with
the exact top-k of q_sel . k ("IceCache", Table 1: the TOP-k row is the exact
top-k; Figure 2 steps 1-2: keys projected on random directions, the query's
pages found by a prioritised search). The pieces of the reading are separated:
  * the MIPS-to-NN transform is exact (the true transformed distance finds the
    exact top-k);
  * the projection: the k nearest in the projected space of one composite's 8
    directions, of both composites' 16, and of more random directions;
  * the search's candidates and the page granularity: no selection of
    budget / P pages can cover more of the top-k than the pages that hold the
    most of it (the ceiling).
The CPU tests check the orderings these facts imply on a small clustered unit.
`python -m tests.test_recall_readings` prints the study at the 36k-token
shape (four units of one layer) that the design notes quote.
"""
import sys

import numpy as np

T_DEFAULT = 256


def _unit(n, centers, seed, group=4):
    rng = np.random.default_rng(seed)
    mu = rng.standard_normal((centers, 128))
    K = (mu[rng.integers(0, centers, n)] + 0.3 * rng.standard_normal((n, 128))).astype(np.float32)
    c = rng.integers(0, centers)
    Q = (mu[c] + 0.3 * rng.standard_normal((group, 128))).astype(np.float32)
    return K, Q


def study(K, Q, T, seed=0, extra_dirs=(32, 64, 128)):
    """Recall of each piece for one unit; returns a dict of fractions."""
    from oracle.oracle import OracleIndex, directions
    out = {}
    qsel = Q[0].copy()
    for g in range(1, Q.shape[0]):
        qsel = (qsel + Q[g]).astype(np.float32)
    s = K.astype(np.float64) @ qsel.astype(np.float64)
    top = set(np.argsort(-s, kind="stable")[:T].tolist())
    ix = OracleIndex(128, 8, 2, 16, seed).build(K, K)
    page_of = ix.page_of()
    for mult in (1, 4):
        ids, npg, tr = ix.select(Q, T, n_cand=mult * T)
        sel = set(np.nonzero(np.isin(page_of, ids[:npg]))[0].tolist())
        out[f"selected pages, n_cand={mult}T"] = len(sel & top) / T
        cand = set()
        for l in range(2):
            order, _ = ix.leaf_order(Q, l, mult * T)
            d0 = ix.dump(l)
            for li in order:
                cand.update(d0["toks"][d0["off"][li]:d0["off"][li + 1]].tolist())
        out[f"search candidates, n_cand={mult}T"] = len(cand & top) / T
        out[f"search candidates |C| / T, n_cand={mult}T"] = len(cand) / T
    _, _, tr = ix.select(Q, T)
    out["tokens attended / T"] = tr["sel_tokens"] / T
    cnt_top = np.bincount(page_of[list(top)], minlength=page_of.max() + 1)
    out["ceiling: best budget/P pages"] = np.sort(cnt_top)[::-1][:T // 16].sum() / T
    c = 2.0 ** ix.e
    n2 = np.sum(K.astype(np.float64) ** 2, 1)
    kt = np.concatenate([K / c, np.sqrt(np.maximum(0, 1 - n2 / c ** 2))[:, None]], 1)
    qt = np.concatenate([qsel / np.linalg.norm(qsel), [0.0]])
    out["true transformed distance"] = len(
        set(np.argsort(np.sum((kt - qt) ** 2, 1), kind="stable")[:T].tolist()) & top) / T
    u = directions(seed, 2, 8, 128).astype(np.float64).reshape(16, 129)
    for m in (8, 16):
        pk, pq = kt @ u[:m].T, qt @ u[:m].T
        d = np.max(np.abs(pk - pq), 1)
        out[f"projected L-inf nearest T, {m} Rademacher dirs"] = len(
            set(np.argsort(d, kind="stable")[:T].tolist()) & top) / T
    rng = np.random.default_rng(seed + 1)
    for m in extra_dirs:
        G = rng.standard_normal((m, 129)) / 16
        d = np.sum((kt @ G.T - qt @ G.T) ** 2, 1)
        out[f"projected L2 nearest T, {m} Gaussian dirs"] = len(
            set(np.argsort(d, kind="stable")[:T].tolist()) & top) / T
    return out


def test_recall_pieces_order(oracle_mod):
    K, Q = _unit(6000, 64, 3)
    r = study(K, Q, 128, extra_dirs=(64,))
    assert r["true transformed distance"] == 1.0  # the transform itself loses nothing
    assert r["selected pages, n_cand=1T"] <= r["ceiling: best budget/P pages"] + 1e-12
    assert r["ceiling: best budget/P pages"] < 1.0  # pages cannot hold all of the top-k
    # more directions see more of the inner-product order than one composite's 8
    assert r["projected L-inf nearest T, 16 Rademacher dirs"] >= r["projected L-inf nearest T, 8 Rademacher dirs"]
    assert r["projected L2 nearest T, 64 Gaussian dirs"] > r["projected L-inf nearest T, 8 Rademacher dirs"]
    # a larger candidate set covers more of the top-k
    assert r["search candidates, n_cand=4T"] >= r["search candidates, n_cand=1T"]


if __name__ == "__main__":
    sys.path.insert(0, ".")
    from semantic_paged_kv_head_gb300 import synth
    w = synth.scaled(synth.WORKLOADS["llama8b_36k"], n_layers=1, n_kv_heads=4)
    keys, values, centers = synth.make_kv(w)
    q = synth.make_queries(w, centers)
    acc = {}
    for h in range(w.n_kv_heads):
        K = keys[0, 0, h].float().numpy()
        Q = q[0, 0, h * w.group:(h + 1) * w.group].float().numpy()
        for k, v in study(K, Q, T_DEFAULT, seed=w.seed).items():
            acc.setdefault(k, []).append(v)
    for k, v in acc.items():
        print(f"{np.mean(v):7.3f}  {k}")

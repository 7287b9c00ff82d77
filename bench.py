"""Decode-step benchmark of the IceCache select + sparse-attention path on GB300.

One step = ice_select + ice_sparse_attn for every unit (layer x KV head) of a
Llama-3.1-8B-shaped decode step at a 36,864-token context (32 layers, 8 KV
heads, 4 query heads per KV head, d = 128, bf16, page_size 16, token budget
256, 8 projections x 2 composite indices). Inputs are synthetic clustered
Gaussian keys (512 centres per unit) and N(0, 1) values, resident in HBM.
L2 is flushed (256 MiB write) between timed steps, outside the events.

Prints one JSON line. Metric: select+attn latency in us per layer (lower is
better), with the achieved HBM bandwidth of the dominant kernel against the
measured copy bandwidth of the GPU.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ice|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import tempfile
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step select+attn latency (µs/layer) & achieved HBM GB/s vs peak, 1 GB300"
UNIT = "us/layer"
WORKLOAD = "llama8b_36k"
FUSED_KERNEL, FUSED_SRC = "select_kernel<fused>", "ice_select.cu"
CLUSTER_KERNEL, CLUSTER_SRC = "select_cluster_kernel<fused>", "ice_select_cluster.cu"


def fused_kernel_of(units, n_composite, cluster_size=None):
    """The kernel of ice_select_attn for a launch of `units` units, by the rule that
    ice_set_cluster_size documents: 8, 4 or 2 blocks per unit (a cluster) up to 19, 38
    or 76 units, one block per unit above, unless a size is set."""
    k = cluster_size if cluster_size else (8 if units <= 19 else 4 if units <= 38 else
                                           2 if units <= 76 else 1)
    if k < n_composite:
        k = 1
    return (CLUSTER_KERNEL, CLUSTER_SRC) if k >= 2 else (FUSED_KERNEL, FUSED_SRC)
FLUSH_BYTES = 256 << 20
INSERT_WORKLOAD = "mistral7b_gen8k"
# the single-replica measurements after the headline, in the order they run
EXTRAS = ("per_layer_serial", "insert", "host_kv", "reuse", "recall")


def leaf_bytes(w):
    """Index bytes per leaf in the canonical count: the cell's low and high code
    of every projection (2m bytes) plus a 4-byte count/offset."""
    return 2 * w.n_proj + 4


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _workload(name):
    from semantic_paged_kv_head_gb300 import synth
    return synth.WORKLOADS[name]


def _config(w):
    return {"workload": w.name, "n_layers": w.n_layers, "n_kv_heads": w.n_kv_heads,
            "group": w.group, "d": w.d, "n_tokens": w.n_tokens, "batch": w.batch,
            "page_size": w.page_size, "token_budget": w.budget, "n_proj": w.n_proj,
            "n_composite": w.n_composite, "n_centers": w.n_centers,
            "l2": "flushed between steps (256 MiB write, outside the timed events)"}


# --------------------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0, out_path=None):
        self.proc = None
        # ICE_BENCH_CLOCKS names a file to keep the raw samples in
        self.path = out_path or os.environ.get("ICE_BENCH_CLOCKS") or os.path.join(
            tempfile.gettempdir(), f"ice_bench_clocks_{os.getpid()}.csv")
        self.dev = device_index

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------------------
# the oracle (CPU) on a bounded sample: cpu_baseline leg and the reference arm
# --------------------------------------------------------------------------------------
def oracle_time_units(w, keys_u, values_u, q_u, budget_s=10.0):
    """Time oracle select+attn over the given units (lists of CPU tensors).
    Returns (us per unit, repetitions, per-unit (page_ids, n_pages, trace))."""
    from oracle.oracle import OracleIndex
    idx = []
    for k, v in zip(keys_u, values_u):
        ix = OracleIndex(w.d, w.n_proj, w.n_composite, w.page_size, w.seed)
        ix.build(k, v)
        idx.append(ix)
    results = []
    for ix, q in zip(idx, q_u):
        ids, npg, tr = ix.select(q, w.budget)
        ix.attn(q, ids, npg)
        results.append((ids, npg, tr))
    reps = 0
    t0 = time.perf_counter()
    while True:
        for ix, q in zip(idx, q_u):
            ids, npg, _ = ix.select(q, w.budget)
            ix.attn(q, ids, npg)
            reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return dt / reps * 1e6, reps, results


def run_reference(args):
    """--impl reference: the oracle as it stands, on the host cores, one layer
    (8 KV-head units) of the same workload shape per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from semantic_paged_kv_head_gb300 import synth
    w = _workload(args.workload)
    ws = synth.scaled(w, n_layers=1, batch=1)
    keys, values, centers = synth.make_kv(ws)
    q = synth.make_queries(ws, centers)
    from oracle.oracle import OracleIndex
    idx, qs = [], []
    for h in range(ws.n_kv_heads):
        ix = OracleIndex(w.d, w.n_proj, w.n_composite, w.page_size, w.seed)
        ix.build(keys[0, 0, h], values[0, 0, h])
        idx.append(ix)
        qs.append(q[0, 0, h * w.group:(h + 1) * w.group])

    def step():
        for ix, qq in zip(idx, qs):
            ids, npg, _ = ix.select(qq, w.budget)
            ix.attn(qq, ids, npg)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    us_layer = dt * 1e6  # one step = one layer (all KV heads)
    sample = (f"one layer ({ws.n_kv_heads} KV-head units, {w.n_tokens} tokens each) of the "
              f"{w.name} shape per step; oracle build untimed")
    line = {"impl": "reference", "metric": METRIC, "value": round(us_layer, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 4), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 select (fixed-order fp32 dot), f64 attention",
            "data": "synthetic", "config": dict(_config(w), l2="not applicable (host oracle)"),
            "cpu_baseline": {"value": round(us_layer, 3), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(us_layer, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------------------
def _traffic_for(kernel, src_file, workload, units):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel and describes this workload at this number of
    units per launch (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent:
        return None
    with open(os.path.join(ROOT, "semantic_paged_kv_head_gb300", "csrc", src_file), "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    if ent.get("source_sha") != h or ent.get("workload") != workload or ent.get("units") != units:
        return None
    return ent.get("dram_bytes_per_launch_full")


def reduce_max(values, device, world):
    """Element-wise maximum over the ranks (the step time of the job is its
    slowest replica); identity with one rank."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def us_per_layer(ms_step, w, world):
    """Whole-job µs per layer: every rank runs a replica of the workload, so one
    step processes world x batch x n_layers layers."""
    return ms_step * 1e3 / (w.n_layers * w.batch * world)


def per_layer_serial(ice, w, keys, values, q, per_step, args, step_bytes, peak):
    """One launch per layer, in sequence, as a decode loop issues them: an index per
    layer (its KV heads), and the step = n_layers fused calls after an L2 flush."""
    import torch
    idx, qs, outs = [], [], []
    for l in range(w.n_layers):
        kl = keys[:, l:l + 1].contiguous()
        vl = values[:, l:l + 1].contiguous()
        idx.append(ice.IceIndex.build(kl, vl, page_size=w.page_size, n_q_heads=w.n_q_heads,
                                      n_composite=w.n_composite, n_proj=w.n_proj, seed=w.seed))
        qs.append(q[:, l:l + 1].contiguous())
        outs.append(torch.empty_like(qs[-1]))
        del kl, vl

    def step(mark):
        for ixl, ql, ol in zip(idx, qs, outs):
            ixl.select_attn(ql, w.budget, ol)

    n = max(20, args.steps)
    per_step(step, 3)
    ms = statistics.median(x[0] for x in per_step(step, n))
    for ixl in idx:
        ixl.check()
        ixl.destroy()
    us = ms * 1e3 / (w.n_layers * w.batch)
    gbs = step_bytes / (ms * 1e-3) / 1e9
    return {"value": round(us, 3), "unit": UNIT, "launches_per_step": w.n_layers,
            "achieved_gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "samples": n,
            "note": (f"each layer's {w.batch * w.n_kv_heads} units in their own launch, the "
                     f"{w.n_layers} launches in sequence after an L2 flush; median of per-step "
                     "event pairs; frac = the step's canonical bytes / time / measured peak")}


def host_kv_run(ice, w, keys, values, q, flush, timed, args, st):
    """The offloaded KV tier: the same workload with the page pool in pinned host
    memory (the index stays in HBM); select+attn latency, the bytes read from
    the pool per step over the CPU-GPU link, and the link's copy bandwidth."""
    import torch
    ix = ice.IceIndex.build(keys, values, page_size=w.page_size, n_q_heads=w.n_q_heads,
                            n_composite=w.n_composite, n_proj=w.n_proj, seed=w.seed, kv_host=True)
    if args.cluster_size is not None:
        ix.set_cluster_size(args.cluster_size)
    out = torch.empty_like(q)
    n = max(20, args.steps // 30)
    timed(lambda: ix.select_attn(q, w.budget, out), 3)
    t_f = timed(lambda: flush.zero_(), n)
    t_s = timed(lambda: (flush.zero_(), ix.select_attn(q, w.budget, out)), n)
    ix.check()
    host_bytes = ix.info().host_bytes
    ix.destroy()
    ms = (t_s - t_f) / n
    es = 2 if w.dtype == torch.bfloat16 else 4
    pool_bytes = st[1] * w.d * es + st[2] * 2 * w.d * es  # rescored key rows + selected pages
    # the link: a pinned host -> device copy of 1 GiB
    hbuf = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(1 << 30, dtype=torch.uint8, device=q.device)
    t_c = timed(lambda: dbuf.copy_(hbuf, non_blocking=True), 5)
    del hbuf, dbuf
    return {"value": round(ms * 1e3 / (w.n_layers * w.batch), 3), "unit": UNIT,
            "pool_bytes_per_step": int(pool_bytes),
            "pool_read_gbs": round(pool_bytes / (ms * 1e-3) / 1e9, 1),
            "link_h2d_copy_gbs": round(5 * (1 << 30) / (t_c * 1e-3) / 1e9, 1),
            "host_pool_bytes": int(host_bytes),
            "note": ("page pool (K and V rows) in pinned host memory mapped into the GPU; "
                     "ice_select + ice_sparse_attn read it over the CPU-GPU link; L2 flushed "
                     "between steps")}


REUSE_R, REUSE_RHO, REUSE_STEPS = 8, 0.995, 64


def reuse_run(ice, synth, ix, w, centers, flush, timed, args):
    """Selection reuse across steps (ice_select_attn_reuse, r = REUSE_R) over a
    stream of correlated decode queries (AR(1) noise, rho = REUSE_RHO)."""
    import torch
    U, n_sel = ix.n_units, w.budget // w.page_size
    qs = synth.make_query_stream(w, centers, REUSE_STEPS, REUSE_RHO)
    ids = torch.full((U, n_sel), -1, dtype=torch.int32, device=centers.device)
    npg = torch.zeros((U,), dtype=torch.int32, device=centers.device)
    out = torch.empty_like(qs[0])
    flags = torch.zeros((REUSE_STEPS, U), dtype=torch.int32, device=centers.device)

    def stream():
        ix.reuse_reset()
        for t in range(REUSE_STEPS):
            flush.zero_()
            ix.select_attn_reuse(qs[t], w.budget, REUSE_R, ids, npg, out, reselected=flags[t])

    def flushes():
        for _ in range(REUSE_STEPS):
            flush.zero_()

    timed(stream, 1)
    reps = max(2, args.steps // 300)
    t_s = timed(stream, reps)
    t_f = timed(flushes, reps)
    ix.check()
    frac = float(flags.float().mean())
    ms = (t_s - t_f) / (reps * REUSE_STEPS)
    return {"value": round(ms * 1e3 / (w.n_layers * w.batch), 4), "unit": UNIT, "r": REUSE_R,
            "reselect_fraction": round(frac, 4), "steps": REUSE_STEPS,
            "note": (f"{REUSE_STEPS} consecutive steps of AR(1)-correlated queries (rho {REUSE_RHO}); "
                     "a unit keeps its pages while its query codes are unchanged, at most r steps; "
                     "L2 flushed between steps; two launches per step (reuse decision, fused "
                     "select+attn)")}


RECALL_NCAND = (1, 2, 4)  # n_cand as multiples of the token budget (shared-memory bound: <= 4x)


def recall_run(ice, w, keys, values, q, flush, timed, args):
    """recall@k (k = the token budget) of the tokens in the selected pages against
    the exact top-k of the group query q_sel . k (fp64 brute force), for one
    layer of the workload and n_cand = 1, 2, 4 x budget; with the latency of
    that layer's fused call (one launch, L2 flushed)."""
    import numpy as np
    import torch
    kl = keys[:, :1].contiguous()
    vl = values[:, :1].contiguous()
    ql = q[:, :1].contiguous()
    U1 = w.batch * w.n_kv_heads
    K = kl.view(U1, w.n_tokens, w.d).float().cpu().numpy().astype(np.float64)
    Q = ql.view(U1, w.group, w.d).float().cpu().numpy()
    k = w.budget
    top = []
    for u in range(U1):
        qs = Q[u].sum(0, dtype=np.float32).astype(np.float64)  # q_sel in fp32, as selected
        sc = K[u] @ qs
        top.append(set(np.argpartition(-sc, k - 1)[:k].tolist()))
    res = []
    out = torch.empty_like(ql)
    for mult in RECALL_NCAND:
        ix = ice.IceIndex.build(kl, vl, page_size=w.page_size, n_q_heads=w.n_q_heads,
                                n_composite=w.n_composite, n_proj=w.n_proj, seed=w.seed,
                                n_cand=mult * w.budget)
        _, ids, npg = ix.select_attn(ql, w.budget, out)
        torch.cuda.synchronize()
        ix.check()
        rec = []
        for u in range(U1):
            c0 = ix.dump(u)["comp"][0]
            sel = set()
            for p in ids[u, :int(npg[u])].tolist():
                sel.update(c0["slot_tok"][p, :c0["list_cnt"][p]].tolist())
            rec.append(len(sel & top[u]) / k)
        n = max(20, args.steps // 50)
        t_f = timed(lambda: flush.zero_(), n)
        t_s = timed(lambda: (flush.zero_(), ix.select_attn(ql, w.budget, out)), n)
        ix.destroy()
        res.append({"n_cand": mult * w.budget, "recall_at_k": round(float(np.mean(rec)), 4),
                    "min_unit": round(float(np.min(rec)), 4),
                    "layer_us": round((t_s - t_f) / n * 1e3, 2)})
    # variants at n_cand = budget: Gaussian directions; per-query-head selection
    # with a union over the group (up to G x budget/P pages attended)
    ix = ice.IceIndex.build(kl, vl, page_size=w.page_size, n_q_heads=w.n_q_heads,
                            n_composite=w.n_composite, n_proj=w.n_proj, seed=w.seed, dir_kind=1)
    _, ids, npg = ix.select_attn(ql, w.budget, out)
    torch.cuda.synchronize()
    ix.check()
    rec = []
    for u in range(U1):
        c0 = ix.dump(u)["comp"][0]
        sel = set()
        for p in ids[u, :int(npg[u])].tolist():
            sel.update(c0["slot_tok"][p, :c0["list_cnt"][p]].tolist())
        rec.append(len(sel & top[u]) / k)
    ix.destroy()
    gauss = {"recall_at_k": round(float(np.mean(rec)), 4), "n_cand": w.budget}
    ix = ice.IceIndex.build(kl, vl, page_size=w.page_size, n_q_heads=w.n_q_heads,
                            n_composite=w.n_composite, n_proj=w.n_proj, seed=w.seed)
    uids, un, _, _ = ix.select_heads(ql, w.budget)
    torch.cuda.synchronize()
    rec, pages = [], []
    for u in range(U1):
        c0 = ix.dump(u)["comp"][0]
        sel = set()
        for p in uids[u, :int(un[u])].tolist():
            sel.update(c0["slot_tok"][p, :c0["list_cnt"][p]].tolist())
        rec.append(len(sel & top[u]) / k)
        pages.append(int(un[u]))
    n = max(20, args.steps // 50)
    t_f = timed(lambda: flush.zero_(), n)

    def heads_step():
        flush.zero_()
        a, b, _, _ = ix.select_heads(ql, w.budget)
        ix.sparse_attn(ql, a, b, out)

    t_s = timed(heads_step, n)
    ix.check()
    ix.destroy()
    heads = {"recall_at_k": round(float(np.mean(rec)), 4), "pages_per_unit": round(float(np.mean(pages)), 1),
             "layer_us": round((t_s - t_f) / n * 1e3, 2),
             "note": "ice_select_heads + ice_sparse_attn over the union, one layer"}
    return {"k": k, "units": U1, "curve": res, "gaussian_directions": gauss, "per_head_union": heads,
            "note": ("tokens of the selected pages against the exact top-k tokens of q_sel (fp64); "
                     "one layer, one launch per n_cand, L2 flushed")}


def insert_run(ice, synth, dev, flush, timed, args):
    """Generation with insertion (the Mistral-7B shape): prefill 8192 tokens, then
    one inserted token per KV head per step for 8192 steps from a drifting
    mixture; insert latency, select+attn latency before and after, leaf growth."""
    import torch
    w = synth.WORKLOADS[INSERT_WORKLOAD]
    keys, values, centers = synth.make_kv(w, device=dev)
    deltas = synth.make_drift(w, centers)
    ks, vs = [], []
    for t in range(w.n_insert):
        k, v = synth.make_insert_token(w, centers, deltas, t)
        ks.append(k)
        vs.append(v)
    K = torch.stack(ks)
    V = torch.stack(vs)
    del ks, vs
    n_graph = 512  # decode steps timed eagerly and as CUDA-graph replays after the inserts
    dec_graph = 16  # decode steps per captured graph
    ins_graph, ins_reps = 64, 10  # inserts per captured graph, replays
    ix = ice.IceIndex.build(keys, values, page_size=w.page_size, n_q_heads=w.n_q_heads,
                            n_composite=w.n_composite, n_proj=w.n_proj, seed=w.seed,
                            max_tokens=w.n_tokens + w.n_insert + 2 * n_graph + ins_graph * (ins_reps + 1) + 8)
    q0 = synth.make_queries(w, centers, step=0, drift_deltas=deltas)
    q1 = synth.make_queries(w, centers, step=w.n_insert, drift_deltas=deltas)
    out = torch.empty_like(q0)
    n_sa = max(50, args.steps // 20)

    def sa_us(qq):
        t_f = timed(lambda: flush.zero_(), n_sa)
        t_s = timed(lambda: (flush.zero_(), ix.select_attn(qq, w.budget, out)), n_sa)
        return (t_s - t_f) / n_sa * 1e3 / (w.n_layers * w.batch)

    U = ix.n_units
    leaves0 = [ix.dump(u)["n_leaf"] for u in range(U)]
    before = sa_us(q0)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(w.n_insert):
        ix.insert(K[t], V[t])
    e1.record()
    torch.cuda.synchronize()
    ix.check()
    us_ins = e0.elapsed_time(e1) * 1e3 / w.n_insert
    after = sa_us(q1)
    ix.check()
    leaves1 = [ix.dump(u)["n_leaf"] for u in range(U)]
    # device time of an insert: a CUDA graph of ins_graph inserts, replayed (the eager
    # loop above is bound by the host's call overhead)
    kg, vg = K[0].clone(), V[0].clone()
    gi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gi):
        for _ in range(ins_graph):
            ix.insert(kg, vg)
    t_ig = timed(gi.replay, ins_reps)
    ix.check()
    n_fin = w.n_tokens + w.n_insert
    # whole decode steps (insert + select + attention): eager calls against the
    # replay of one step captured in a CUDA graph
    ids = torch.empty((U, w.budget // w.page_size), dtype=torch.int32, device=dev)
    npg = torch.empty((U,), dtype=torch.int32, device=dev)
    ks, vs = K[0].clone(), V[0].clone()
    t_eager = timed(lambda: ix.decode_step(ks, vs, q1, w.budget, ids, npg, out), n_graph)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(dec_graph):
            ix.decode_step(ks, vs, q1, w.budget, ids, npg, out)
    t_graph = timed(g.replay, n_graph // dec_graph)
    ix.check()
    pages0 = sum(x[0] for x in leaves0)
    pages1 = sum(x[0] for x in leaves1)
    ix.destroy()
    return {"workload": w.name, "units": U, "steps": w.n_insert,
            "insert_us_per_step": round(t_ig / (ins_reps * ins_graph) * 1e3, 3),
            "insert_us_per_step_eager": round(us_ins, 3),
            "note": ("one ice_insert call per step inserts one token into every unit; device time "
                     f"per call from replays of a CUDA graph of {ins_graph} calls (no L2 flush); "
                     "_eager: back-to-back calls from Python, bound by the host's call overhead"),
            "select_attn_us_per_layer_before": round(before, 3),
            "select_attn_us_per_layer_after": round(after, 3),
            "pages_per_unit_before": round(pages0 / U, 1), "pages_per_unit_after": round(pages1 / U, 1),
            "occupancy_before": round(w.n_tokens * U / (pages0 * w.page_size), 4),
            "occupancy_after": round(n_fin * U / (pages1 * w.page_size), 4),
            "leaves_per_unit_after": [round(sum(x[l] for x in leaves1) / U, 1)
                                      for l in range(w.n_composite)],
            "decode_step_us": {"eager": round(t_eager / n_graph * 1e3, 3),
                               "cuda_graph": round(t_graph / n_graph * 1e3, 3),
                               "note": ("ice_decode_step (insert + fused select/attention, all units) "
                                        "back to back, no L2 flush; eager calls vs replays of a "
                                        f"graph of {dec_graph} captured steps (per step)")}}


def _oracle_worker(a):
    """One process of the parallel oracle timing: build untimed, then time
    select+attn of its unit for the given wall budget."""
    d, m, L, P, seed, budget, k, v, qq, secs = a
    from oracle.oracle import OracleIndex
    ix = OracleIndex(d, m, L, P, seed)
    ix.build(k, v)
    ids, npg, _ = ix.select(qq, budget)
    ix.attn(qq, ids, npg)
    reps = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < secs:
        ids, npg, _ = ix.select(qq, budget)
        ix.attn(qq, ids, npg)
        reps += 1
    return (time.perf_counter() - t0) / max(reps, 1)


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_parallel(w, keys, values, q, U, args):
    """The oracle over independent units in nproc processes (spawned)."""
    import multiprocessing as mp
    nproc = os.cpu_count() or 1
    units = [(i * U) // nproc for i in range(nproc)]
    secs = max(2.0, args.cpu_seconds / 2)
    jobs = []
    for u in units:
        k = keys.view(U, w.n_tokens, w.d)[u].float().cpu().numpy()
        v = values.view(U, w.n_tokens, w.d)[u].float().cpu().numpy()
        qq = q.view(U, w.group, w.d)[u].float().cpu().numpy()
        jobs.append((w.d, w.n_proj, w.n_composite, w.page_size, w.seed, w.budget, k, v, qq, secs))
    t0 = time.perf_counter()
    with mp.get_context("spawn").Pool(nproc) as pool:
        per = pool.map(_oracle_worker, jobs)
    wall = time.perf_counter() - t0
    units_per_layer = U // (w.n_layers * w.batch)
    # nproc units in flight at once: throughput nproc / mean(seconds per unit)
    us_layer = statistics.mean(per) * 1e6 * units_per_layer / nproc
    return {"value": round(us_layer, 2), "unit": UNIT, "cores": nproc, "kind": "oracle",
            "cpu": _cpu_model(), "wall_s": round(wall, 1),
            "sample": (f"{nproc} units of this workload, one per process, each timed for "
                       f"~{secs:.0f} s; build untimed")}


def run_ice(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from semantic_paged_kv_head_gb300 import build as ice_build
    ice_build.build_lib()
    from semantic_paged_kv_head_gb300 import ice, synth

    w = _workload(args.workload)
    if args.layers:
        w = synth.scaled(w, n_layers=args.layers)
    dev = torch.device("cuda", local)
    keys, values, centers = synth.make_kv(w, device=dev)
    q = synth.make_queries(w, centers)
    # a small build first, so that the timed build does not include the library's
    # one-time setup (kernel attributes, the driver's tensor-map encoder)
    ice.IceIndex.build(keys[:, :1, :1, :1024].contiguous(), values[:, :1, :1, :1024].contiguous(),
                       page_size=w.page_size, n_q_heads=w.group, n_composite=w.n_composite,
                       n_proj=w.n_proj, seed=w.seed).destroy()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ix = ice.IceIndex.build(keys, values, page_size=w.page_size, n_q_heads=w.n_q_heads,
                            n_composite=w.n_composite, n_proj=w.n_proj, seed=w.seed)
    torch.cuda.synchronize()
    build_ms = (time.perf_counter() - t0) * 1e3
    if args.cluster_size is not None:
        ix.set_cluster_size(args.cluster_size)
    U = ix.n_units
    n_sel = w.budget // w.page_size
    page_ids = torch.empty((U, n_sel), dtype=torch.int32, device=dev)
    n_pages = torch.empty((U,), dtype=torch.int32, device=dev)
    stats = torch.zeros((U, 4), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    # canonical algorithmic bytes of a step (counters verified against the oracle
    # trace by the tests): per leaf 2m + 4 B (cell low/high codes, count/offset),
    # per rescored candidate its key row + 4 B id, per token of a selected page its
    # K and V rows, per unit the G query rows in and the G output rows out
    ix.select(q, w.budget, page_ids, n_pages, stats)
    ix.sparse_attn(q, page_ids, n_pages, out)
    torch.cuda.synchronize()
    ix.check()
    st = stats.double().sum(0).tolist()
    es = 2 if w.dtype == torch.bfloat16 else 4
    q_b = U * w.group * w.d * es
    sel_bytes = st[0] * leaf_bytes(w) + st[1] * (w.d * es + 4) + q_b
    attn_bytes = st[2] * 2 * w.d * es + 2 * q_b
    step_bytes = sel_bytes + attn_bytes - q_b  # the fused step reads q once

    def flush_only():
        flush.zero_()

    def flush_fused():
        flush.zero_()
        ix.select_attn(q, w.budget, out, page_ids, n_pages)

    def per_step(fn, k, flush_first=True, marks=2):
        """Device time of each of k steps: the L2 flush (outside the events), then
        CUDA events on the launching stream around the step's launches. fn(mark)
        runs the step and calls mark() between its parts (marks - 2 times)."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(marks)] for _ in range(k)]
        torch.cuda.synchronize()
        for i in range(k):
            if flush_first:
                flush.zero_()
            it = iter(ev[i])
            next(it).record(stream)
            fn(lambda: next(it).record(stream))
            next(it).record(stream)
        torch.cuda.synchronize()
        return [[e[j].elapsed_time(e[j + 1]) for j in range(marks - 1)] for e in ev]

    def fused_step(mark):
        ix.select_attn(q, w.budget, out, page_ids, n_pages)

    def separate_step(mark):
        ix.select(q, w.budget, page_ids, n_pages)
        mark()
        ix.sparse_attn(q, page_ids, n_pages, out)

    warm_n = max(3, args.warmup)
    per_step(fused_step, warm_n)
    per_step(separate_step, warm_n, marks=3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # the timed region: exactly args.steps fused steps (one launch each), every
    # step after an L2 flush and bracketed by its own pair of events
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        fused_ms = [x[0] for x in per_step(fused_step, args.steps)]
        wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    n_steps = args.steps

    def pct(xs, f):
        xs = sorted(xs)
        return xs[min(len(xs) - 1, max(0, int(round(f * (len(xs) - 1)))))]

    ms_fused = statistics.median(fused_ms)
    fused_p10, fused_p90 = pct(fused_ms, 0.1), pct(fused_ms, 0.9)
    # the two separate calls, the same number of steps, each call between events
    sep = per_step(separate_step, args.steps, marks=3)
    ms_sel = statistics.median([x[0] for x in sep])
    ms_att = statistics.median([x[1] for x in sep])
    ms_sep = statistics.median([x[0] + x[1] for x in sep])
    # cross-check: back-to-back loops by subtraction, [flush + step] - [flush]
    def timed(fn, k):
        """Device time of k back-to-back calls (the host runs ahead of the GPU)."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    n_x = max(50, args.steps)
    ms_loop = (timed(flush_fused, n_x) - timed(flush_only, n_x)) / n_x
    (ms_sel, ms_att, ms_sep, ms_fused, fused_p10, fused_p90,
     ms_loop) = reduce_max([ms_sel, ms_att, ms_sep, ms_fused, fused_p10, fused_p90, ms_loop], dev,
                           world)
    ms_step = ms_fused  # the reported path is always the fused call (one launch per step)
    ix.check()

    # end to end through the public API with host buffers, every step: q in page-locked
    # host memory, the result back in page-locked host memory. (a) the call reads q and
    # writes out in place over the CPU-GPU link; (b) explicit copies around the call.
    q_host = q.cpu().pin_memory()
    out_host = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    q_in = torch.empty_like(q)
    n_e2e = max(20, args.steps)

    def e2e_loop(step):
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_e2e)]
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        for k in range(n_e2e):
            flush.zero_()
            ev2[k][0].record(stream)
            step()
            ev2[k][1].record(stream)
        torch.cuda.synchronize()
        return reduce_max([statistics.median(e[0].elapsed_time(e[1]) for e in ev2)], dev, world)[0]

    def step_in_place():
        ix.select_attn(q_host, w.budget, out_host, page_ids, n_pages)

    def step_copies():
        q_in.copy_(q_host, non_blocking=True)
        ix.select_attn(q_in, w.budget, out, page_ids, n_pages)
        out_host.copy_(out, non_blocking=True)

    ms_e2e = e2e_loop(step_in_place)
    torch.cuda.synchronize()
    ref_out = out_host.clone()
    ms_e2e_copies = e2e_loop(step_copies)
    torch.cuda.synchronize()
    if not torch.equal(ref_out, out_host):
        raise RuntimeError("in-place host-buffer call and the copied call disagree")

    peak, peak_kind = _peaks()
    sel_gbs = sel_bytes / (ms_sel * 1e-3) / 1e9
    att_gbs = attn_bytes / (ms_att * 1e-3) / 1e9
    # the reported path is always the fused call; it is one kernel, so the roofline
    # kernel is that kernel and its time is the step's
    dom, src = fused_kernel_of(U, w.n_composite, args.cluster_size)
    dom_bytes, dom_ms = step_bytes, ms_fused
    dom_gbs = dom_bytes / (dom_ms * 1e-3) / 1e9
    # every rank runs its own replica of the workload: the job processes
    # world x n_layers layers per step
    us_layer = us_per_layer(ms_step, w, world)
    line = {
        "metric": METRIC, "value": round(us_layer, 4), "unit": UNIT, "n_gpus": world,
        "steps": n_steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": _config(w),
        "step_bytes": int(step_bytes),
        "step_gbs": round(step_bytes / (ms_step * 1e-3) / 1e9, 1),
        "step_frac_of_peak": round(step_bytes / (ms_step * 1e-3) / 1e9 / peak, 4),
        "path": "ice_select_attn (select and paged attention fused, one launch per step)",
        "step_us": {"median": round(ms_fused * 1e3, 3), "p10": round(fused_p10 * 1e3, 3),
                    "p90": round(fused_p90 * 1e3, 3), "samples": n_steps,
                    "loop_crosscheck": round(ms_loop * 1e3, 3), "loop_steps": n_x},
        "kernels": {dom: {"us": round(ms_fused * 1e3, 3),
                                             "bytes": int(step_bytes),
                                             "gbs": round(step_bytes / (ms_fused * 1e-3) / 1e9, 1)},
                    "separate_calls": {"us": round(ms_sep * 1e3, 3),
                                       "select_us": round(ms_sel * 1e3, 3),
                                       "select_gbs": round(sel_gbs, 1),
                                       "attn_us": round(ms_att * 1e3, 3),
                                       "attn_gbs": round(att_gbs, 1)}},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(dom_gbs, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                     "traffic": _traffic_for(dom, src, w.name, U), "algorithmic_bytes": int(dom_bytes)},
        "e2e": {"value": round(us_per_layer(ms_e2e, w, world), 4), "unit": UNIT,
                "h2d_bytes_per_step": int(q.numel() * q.element_size()),
                "d2h_bytes_per_step": int(out.numel() * out.element_size()),
                "how": ("ice_select_attn on page-locked host q and out: the kernel reads q and "
                        "writes the result over the CPU-GPU link; L2 flushed before each step"),
                "with_copies": {"value": round(us_per_layer(ms_e2e_copies, w, world), 4),
                                "unit": UNIT, "how": "cudaMemcpyAsync of q in and out back "
                                "around ice_select_attn on device buffers"}},
        "gpu_launches": n_steps,
        "timing": ("median over the timed steps of each step's own CUDA-event pair on the "
                   "launching stream; every step follows an L2 flush (256 MiB write) outside its "
                   "events; p10/p90 over the same steps; loop_crosscheck = ([flush + step] - "
                   "[flush]) over back-to-back loops of loop_steps steps; separate calls timed "
                   "per call with events over the same number of steps"),
        "build_ms": round(build_ms, 1),
        "wall_s_timed_region": round(wall, 3),
        "clocks": clk.summary(),
    }
    # warm L2 (no flush): the same fused step, each step between its own events
    n_w = max(50, args.steps)
    t_w = statistics.median(x[0] for x in per_step(fused_step, n_w, flush_first=False))
    t_w = reduce_max([t_w], dev, world)[0]
    line["warm"] = {"value": round(us_per_layer(t_w, w, world), 4), "unit": UNIT,
                    "samples": n_w,
                    "note": "no L2 flush between steps; median of per-step event pairs"}
    if not args.no_extras and world == 1:  # single-replica extras (not part of scaling runs)
        runs = {
            "per_layer_serial": lambda: per_layer_serial(ice, w, keys, values, q, per_step, args,
                                                         step_bytes, peak),
            "insert": lambda: insert_run(ice, synth, dev, flush, timed, args),
            "host_kv": lambda: host_kv_run(ice, w, keys, values, q, flush, timed, args, st),
            "reuse": lambda: reuse_run(ice, synth, ix, w, centers, flush, timed, args),
            "recall": lambda: recall_run(ice, w, keys, values, q, flush, timed, args),
        }
        chosen = [e for e in args.extras.split(",") if e]  # names checked when parsing
        for name in EXTRAS:
            if name in chosen:
                # an NVTX range per extra, so that a profiler can take the launches of one
                torch.cuda.nvtx.range_push(name)
                line[name] = runs[name]()
                torch.cuda.synchronize()
                torch.cuda.nvtx.range_pop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample_units = sorted({0, U // 3, (2 * U) // 3, U - 1})
        ku = [keys.view(U, w.n_tokens, w.d)[u].cpu() for u in sample_units]
        vu = [values.view(U, w.n_tokens, w.d)[u].cpu() for u in sample_units]
        qu = [q.view(U, w.group, w.d)[u].cpu() for u in sample_units]
        us_unit, reps, res = oracle_time_units(w, ku, vu, qu, budget_s=args.cpu_seconds)
        units_per_layer = U // (w.n_layers * w.batch)
        ids_cpu = page_ids.cpu().numpy()
        same = all(res[i][1] == int(n_pages[u]) and
                   (ids_cpu[u][:n_sel] == res[i][0]).all() for i, u in enumerate(sample_units))
        st_cpu = stats.cpu().numpy()
        stats_same = all(st_cpu[u][0] == res[i][2]["leaves"] and st_cpu[u][1] == res[i][2]["cands"]
                         and st_cpu[u][2] == res[i][2]["sel_tokens"]
                         for i, u in enumerate(sample_units))
        line["cpu_baseline"] = {
            "value": round(us_unit * units_per_layer, 2), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": (f"units {sample_units} of this workload, select+attn repeated {reps} times "
                       f"(~{args.cpu_seconds:.0f} s, single thread); oracle build untimed; "
                       f"us/layer = us/unit x {units_per_layer} KV heads")}
        line["parity_sampled"] = {"units": sample_units, "page_ids_equal": bool(same),
                                  "byte_counters_equal": bool(stats_same)}
        if not args.no_extras:
            line["cpu_baseline_parallel"] = oracle_parallel(w, keys, values, q, U, args)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ice", "reference"], default="ice")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--cluster-size", type=int, default=None,
                    help="blocks per unit of the selection (0 automatic; profiling)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-layer-serial, insert and parallel-oracle measurements")
    ap.add_argument("--extras", default=",".join(EXTRAS),
                    help="comma list of the extras to run (profiling one of them): " + ",".join(EXTRAS))
    args = ap.parse_args()
    unknown = [e for e in args.extras.split(",") if e and e not in EXTRAS]
    if unknown:
        ap.error(f"unknown extra(s) {','.join(unknown)}; choose from {','.join(EXTRAS)}")
    if args.impl == "reference":
        return run_reference(args)
    return run_ice(args)


if __name__ == "__main__":
    sys.exit(main())

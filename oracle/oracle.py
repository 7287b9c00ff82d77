"""Python wrapper of the CPU oracle (test infrastructure only).

The oracle is a plain, single-threaded C++ statement of the IceCache
decode-time path (DCI-tree build, insertion, P-DCI page selection and sparse
GQA attention; "IceCache", Figure 2 and Figure 3). Only the tests, the smoke
check and the benchmark's CPU-baseline leg import this module. It never imports
the GPU package and the GPU package never imports it.

Arrays cross the boundary as numpy arrays. Keys, values and queries are given
as float32; bf16 data is widened here, exactly, by placing its 16 bits in the
high half of a float32.

One oracle object holds the index of ONE unit (one sequence, layer and KV
head).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ice_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None

I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
I64P = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
U64P = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")
U32P = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
F32P = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build_oracle(force: bool = False) -> str:
    """Compile the oracle into oracle/liboracle.so (plain g++, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build_oracle()
    lib = ctypes.CDLL(_LIB)
    vp, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    sig = {
        "orc_splitmix64": (u64, [ctypes.POINTER(ctypes.c_uint64)]),
        "orc_dot": (f32, [F32P, F32P, i32]),
        "orc_scale_exponent": (i32, [f32]),
        "orc_quantise": (i32, [f32]),
        "orc_morton": (u64, [I32P, i32]),
        "orc_directions": (None, [u64, i32, i32, i32, F32P]),
        "orc_create": (vp, [i32, i32, i32, i32, u64]),
        "orc_create_kind": (vp, [i32, i32, i32, i32, u64, i32]),
        "orc_directions_gauss": (None, [u64, i32, i32, i32, F32P]),
        "orc_destroy": (None, [vp]),
        "orc_build": (i32, [vp, F32P, F32P, i32, i32]),
        "orc_insert": (i32, [vp, F32P, F32P]),
        "orc_e": (i32, [vp]),
        "orc_n": (i32, [vp]),
        "orc_n_leaves": (i32, [vp, i32]),
        "orc_next_id": (i32, [vp, i32]),
        "orc_token_keys": (None, [vp, i32, U64P, I32P]),
        "orc_projections": (None, [vp, F32P]),
        "orc_transformed_key": (None, [vp, i32, F32P]),
        "orc_dump": (None, [vp, i32, I32P, U64P, U32P, I32P, I32P, I32P, I32P, I64P, I32P]),
        "orc_query": (None, [vp, F32P, i32, I32P, F32P]),
        "orc_leaf_order": (i32, [vp, F32P, i32, i32, i32, i32, I32P, ctypes.c_void_p]),
        "orc_select": (i32, [vp, F32P, i32, i32, i32, I32P, I32P, I64P, i32]),
        "orc_attn": (None, [vp, F32P, i32, I32P, i32, F64P]),
        "orc_dense_attn": (None, [F32P, i32, F32P, F32P, i32, i32, F64P]),
        "orc_brute_rank": (None, [vp, F32P, i32, I32P]),
        "orc_exact_topk": (None, [vp, F32P, i32, i32, I32P]),
        "orc_page_of": (None, [vp, I32P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def as_f32(x) -> np.ndarray:
    """float32 view of a torch tensor / numpy array; bf16 is widened exactly."""
    if isinstance(x, np.ndarray) or type(x).__module__.split(".")[0] != "torch":
        return np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                bits = x.contiguous().view(torch.int16).numpy().astype(np.uint16)
                return np.ascontiguousarray((bits.astype(np.uint32) << 16).view(np.float32))
            return np.ascontiguousarray(x.to(torch.float32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def splitmix64_stream(seed: int, count: int) -> list[int]:
    lib = _load()
    st = ctypes.c_uint64(seed)
    return [int(lib.orc_splitmix64(ctypes.byref(st))) for _ in range(count)]


def dot(a, b) -> float:
    a, b = as_f32(a).ravel(), as_f32(b).ravel()
    return float(_load().orc_dot(a, b, a.size))


def scale_exponent(maxn: float) -> int:
    return int(_load().orc_scale_exponent(float(maxn)))


def quantise(p: float) -> int:
    return int(_load().orc_quantise(float(p)))


def morton(codes) -> int:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.int32))
    return int(_load().orc_morton(c, c.size))


def directions(seed: int, L: int, m: int, d: int, kind: int = 0) -> np.ndarray:
    """Projection directions [L, m, d+1]: kind 0 Rademacher +-1/16, kind 1 Gaussian."""
    out = np.zeros((L, m, d + 1), dtype=np.float32)
    if kind == 0:
        _load().orc_directions(seed, L, m, d, out.reshape(-1))
    else:
        _load().orc_directions_gauss(seed, L, m, d, out.reshape(-1))
    return out


def dense_attn(q, K, V) -> np.ndarray:
    q, K, V = as_f32(q), as_f32(K), as_f32(V)
    G, d = q.shape
    n = K.shape[0]
    out = np.zeros((G, d), dtype=np.float64)
    _load().orc_dense_attn(q.reshape(-1), G, K.reshape(-1), V.reshape(-1), n, d, out.reshape(-1))
    return out


class OracleIndex:
    """The index of one unit, built by the oracle."""

    def __init__(self, d: int, m: int, L: int, page_size: int, seed: int, dir_kind: int = 0):
        self._lib = _load()
        self.d, self.m, self.L, self.P = d, m, L, page_size
        self._h = self._lib.orc_create_kind(d, m, L, page_size, seed, dir_kind)
        if not self._h:
            raise ValueError("invalid oracle parameters")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.orc_destroy(h)
            self._h = None

    # -- build / insert ---------------------------------------------------
    def build(self, K, V, forced_e: int | None = None):
        K, V = as_f32(K), as_f32(V)
        n = K.shape[0]
        self._lib.orc_build(self._h, K.reshape(-1), V.reshape(-1), n,
                            -(1 << 20) if forced_e is None else int(forced_e))
        return self

    def insert(self, k, v):
        k, v = as_f32(k).ravel(), as_f32(v).ravel()
        self._lib.orc_insert(self._h, k, v)

    # -- inspection -------------------------------------------------------
    @property
    def e(self) -> int:
        return int(self._lib.orc_e(self._h))

    @property
    def n(self) -> int:
        return int(self._lib.orc_n(self._h))

    def n_leaves(self, l: int) -> int:
        return int(self._lib.orc_n_leaves(self._h, l))

    def next_id(self, l: int) -> int:
        return int(self._lib.orc_next_id(self._h, l))

    def token_keys(self, l: int):
        n = self.n
        mk = np.zeros(n, dtype=np.uint64)
        codes = np.zeros((n, self.m), dtype=np.int32)
        self._lib.orc_token_keys(self._h, l, mk, codes.reshape(-1))
        return mk, codes

    def projections(self) -> np.ndarray:
        out = np.zeros((self.n, self.L, self.m), dtype=np.float32)
        self._lib.orc_projections(self._h, out.reshape(-1))
        return out

    def transformed_key(self, t: int) -> np.ndarray:
        out = np.zeros(self.d + 1, dtype=np.float32)
        self._lib.orc_transformed_key(self._h, t, out)
        return out

    def dump(self, l: int) -> dict:
        """Leaves of composite l, left to right (see orc_dump)."""
        N = self.n_leaves(l)
        m = self.m
        t = np.zeros(N, np.int32)
        pm = np.zeros(N, np.uint64)
        pt = np.zeros(N, np.uint32)
        ids = np.zeros(N, np.int32)
        cnt = np.zeros(N, np.int32)
        lo = np.zeros((N, m), np.int32)
        hi = np.zeros((N, m), np.int32)
        off = np.zeros(N + 1, np.int64)
        toks = np.zeros(max(self.n, 1), np.int32)
        self._lib.orc_dump(self._h, l, t, pm, pt, ids, cnt, lo.reshape(-1), hi.reshape(-1), off, toks)
        return {"t": t, "pm": pm, "pt": pt, "id": ids, "cnt": cnt, "lo": lo, "hi": hi,
                "off": off, "toks": toks[: self.n]}

    def page_of(self) -> np.ndarray:
        out = np.zeros(self.n, np.int32)
        self._lib.orc_page_of(self._h, out)
        return out

    # -- query side ---------------------------------------------------------
    def query(self, q):
        q = as_f32(q)
        G = q.shape[0]
        codes = np.zeros((self.L, self.m), np.int32)
        qsel = np.zeros(self.d, np.float32)
        self._lib.orc_query(self._h, q.reshape(-1), G, codes.reshape(-1), qsel)
        return codes, qsel

    def leaf_order(self, q, l: int, n_cand: int, tree: bool = False):
        q = as_f32(q)
        G = q.shape[0]
        N = self.n_leaves(l)
        out = np.zeros(max(N, 1), np.int32)
        prio = np.zeros(max(N, 1), np.int32)
        k = self._lib.orc_leaf_order(self._h, q.reshape(-1), G, l, n_cand, 1 if tree else 0, out,
                                     prio.ctypes.data_as(ctypes.c_void_p))
        return out[:k], prio[:N]

    def select(self, q, budget: int, n_cand: int | None = None, check_tree: bool = False):
        """Returns (page_ids [budget/P] with -1 padding, n_pages, trace dict)."""
        q = as_f32(q)
        G = q.shape[0]
        n_sel = budget // self.P
        ids = np.zeros(max(n_sel, 1), np.int32)
        npg = np.zeros(1, np.int32)
        tr = np.zeros(8, np.int64)
        self._lib.orc_select(self._h, q.reshape(-1), G, budget, budget if n_cand is None else n_cand,
                             ids, npg, tr, 1 if check_tree else 0)
        trace = {"leaves": int(tr[0]), "cands": int(tr[1]), "sel_tokens": int(tr[2]),
                 "tree_ok": bool(tr[3])}
        return ids[:n_sel], int(npg[0]), trace

    def attn(self, q, page_ids, n_pages: int) -> np.ndarray:
        q = as_f32(q)
        G = q.shape[0]
        ids = np.ascontiguousarray(np.asarray(page_ids, dtype=np.int32))
        out = np.zeros((G, self.d), np.float64)
        self._lib.orc_attn(self._h, q.reshape(-1), G, ids, int(n_pages), out.reshape(-1))
        return out

    def brute_rank(self, q) -> np.ndarray:
        q = as_f32(q)
        out = np.zeros(self.n, np.int32)
        self._lib.orc_brute_rank(self._h, q.reshape(-1), q.shape[0], out)
        return out

    def exact_topk(self, q, k: int) -> np.ndarray:
        q = as_f32(q)
        k = min(k, self.n)
        out = np.zeros(max(k, 1), np.int32)
        self._lib.orc_exact_topk(self._h, q.reshape(-1), q.shape[0], k, out)
        return out[:k]


class ReuseOracle:
    """Selection reuse across decode steps ("IceCache" paper, the IceCache(r)
    variant; the paper names it but gives no mechanism).

    Reading: a unit keeps the pages of its last selection for up to r further
    steps while its query codes (``OracleIndex.query``: the 8-bit codes of the
    group query on every projection direction) are exactly those of the step
    that selected them. A changed code, r reuses in a row, no selection yet or
    a changed budget selects again. The attention always reads the kept pages'
    current tokens (inserted tokens included).
    """

    def __init__(self, index: OracleIndex, r: int):
        if r < 0:
            raise ValueError("r must be >= 0")
        self.ix = index
        self.r = r
        self.codes = None
        self.age = -1
        self.budget = None
        self.ids = None
        self.npg = 0

    def step(self, q, budget: int, n_cand: int | None = None):
        """One decode step: returns (page_ids, n_pages, reselected, attention)."""
        codes, _ = self.ix.query(q)
        keep = (self.codes is not None and self.budget == budget and 0 <= self.age < self.r
                and np.array_equal(codes, self.codes))
        if keep:
            self.age += 1
        else:
            self.ids, self.npg, _ = self.ix.select(q, budget, n_cand)
            self.codes = codes
            self.budget = budget
            self.age = 0
        return self.ids, self.npg, not keep, self.ix.attn(q, self.ids, self.npg)


def select_heads(index: OracleIndex, q, budget: int, n_cand: int | None = None):
    """Per-query-head selection with a union over the group (a variant of the
    selection, "IceCache" Figure 2 step 2): head g selects with its own query
    as q_sel; the union lists head 0's pages in order, then every later head's
    pages not listed yet. Returns (union ids, n, per-head [(ids, n)])."""
    q = as_f32(q)
    heads = [index.select(q[g:g + 1], budget, n_cand)[:2] for g in range(q.shape[0])]
    union = []
    for ids, n in heads:
        for p in ids[:n].tolist():
            if p not in union:
                union.append(p)
    return np.asarray(union, dtype=np.int32), len(union), heads

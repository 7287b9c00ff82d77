"""ctypes binding of libice.so (the C ABI declared in include/ice.h).

Argument marshalling only: torch supplies device memory (or, for the decode-step
calls, page-locked CPU tensors that the kernels read and write in place) and the
current CUDA stream; every step of the decode path runs in the library's CUDA
kernels.
There is no CPU fallback. If libice.so is missing or cannot be loaded the
import of this module raises.

    from semantic_paged_kv_head_gb300 import ice
    ix = ice.IceIndex.build(keys, values, page_size=16, n_q_heads=32, n_composite=2)
    page_ids, n_pages = ix.select(q, token_budget=256)
    out = ix.sparse_attn(q, page_ids, n_pages)
    ix.insert(k_new, v_new)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libice.so")

ICE_OK = 0
ICE_ERR_INVALID_ARG = -1
ICE_ERR_CAPACITY = -2
ICE_ERR_CUDA = -3
ICE_ERR_TIMEOUT = -4
ICE_ERR_BOUNDS = -5
ICE_ERR_UNSUPPORTED = -6
ICE_F32 = 0
ICE_BF16 = 1

# every symbol include/ice.h declares
EXPORTS = ["ice_build", "ice_insert", "ice_select", "ice_select_attn", "ice_sparse_attn", "ice_get_error",
           "ice_destroy", "ice_status_string", "ice_get_info", "ice_debug_dump", "ice_debug_page",
           "ice_key_codes_noalloc", "ice_select_attn_reuse", "ice_reuse_reset",
           "ice_debug_set_flags", "ice_select_heads", "ice_decode_step", "ice_set_cluster_size"]


class ice_params(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("n_proj", ctypes.c_int32), ("n_composite", ctypes.c_int32),
                ("n_cand", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("max_tokens", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("kv_location", ctypes.c_int32), ("dir_kind", ctypes.c_int32)]


DIR_RADEMACHER, DIR_GAUSSIAN = 0, 1  # ice_params.dir_kind
KV_DEVICE, KV_HOST = 0, 1  # ice_params.kv_location
DEBUG_STALL_ATTN = 1       # ice_debug_set_flags


class ice_info(ctypes.Structure):
    _fields_ = [("n_units", ctypes.c_int64), ("n_tokens", ctypes.c_int64),
                ("max_tokens", ctypes.c_int64), ("list_capacity", ctypes.c_int64),
                ("pool_bytes", ctypes.c_int64), ("group", ctypes.c_int32),
                ("n_composite", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("host_bytes", ctypes.c_int64),
                ("kv_location", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class IceError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})" if what else status_string(code))


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libice.so and declare the signatures of include/ice.h."""
    if not os.path.exists(path):
        raise ImportError(f"libice.so not built ({path}); run semantic_paged_kv_head_gb300/build.py")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P = ctypes.POINTER
    lib.ice_build.argtypes = [P(ice_params), vp, vp, i64, vp, P(vp)]
    lib.ice_build.restype = ctypes.c_int
    lib.ice_insert.argtypes = [vp, vp, vp, vp]
    lib.ice_insert.restype = ctypes.c_int
    lib.ice_select.argtypes = [vp, vp, i32, vp, vp, vp, vp]
    lib.ice_select.restype = ctypes.c_int
    lib.ice_select_attn.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
    lib.ice_select_attn.restype = ctypes.c_int
    lib.ice_sparse_attn.argtypes = [vp, vp, vp, vp, i32, vp, vp]
    lib.ice_sparse_attn.restype = ctypes.c_int
    lib.ice_get_error.argtypes = [vp, vp]
    lib.ice_get_error.restype = ctypes.c_int
    lib.ice_destroy.argtypes = [vp]
    lib.ice_destroy.restype = None
    lib.ice_status_string.argtypes = [ctypes.c_int]
    lib.ice_status_string.restype = ctypes.c_char_p
    lib.ice_get_info.argtypes = [vp, P(ice_info)]
    lib.ice_get_info.restype = ctypes.c_int
    lib.ice_debug_dump.argtypes = [vp, i32, vp, i64, vp]
    lib.ice_debug_dump.restype = i64
    lib.ice_debug_page.argtypes = [vp, i32, i32, vp, vp, vp]
    lib.ice_debug_page.restype = ctypes.c_int
    lib.ice_key_codes_noalloc.argtypes = [P(ice_params), vp, i64, vp, vp, vp]
    lib.ice_key_codes_noalloc.restype = ctypes.c_int
    lib.ice_select_attn_reuse.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp]
    lib.ice_select_attn_reuse.restype = ctypes.c_int
    lib.ice_reuse_reset.argtypes = [vp, vp]
    lib.ice_reuse_reset.restype = ctypes.c_int
    lib.ice_decode_step.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp]
    lib.ice_decode_step.restype = ctypes.c_int
    lib.ice_select_heads.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
    lib.ice_select_heads.restype = ctypes.c_int
    lib.ice_debug_set_flags.argtypes = [vp, i32]
    lib.ice_debug_set_flags.restype = ctypes.c_int
    lib.ice_set_cluster_size.argtypes = [vp, i32]
    lib.ice_set_cluster_size.restype = ctypes.c_int
    return lib


_lib = load_library()


def status_string(code: int) -> str:
    return _lib.ice_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != ICE_OK:
        raise IceError(code, what)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev_ptr(t: torch.Tensor, dtype=None, name="tensor", host_ok=True) -> int:
    """Address of a buffer argument: a CUDA tensor or, where the call allows it,
    a page-locked CPU tensor that the kernels read or write in place."""
    ok = isinstance(t, torch.Tensor) and (
        t.is_cuda or (host_ok and t.device.type == "cpu" and t.is_pinned()))
    if not ok:
        raise ValueError(f"{name} must be a CUDA tensor" + (" or page-locked CPU tensor" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _like(t: torch.Tensor) -> torch.Tensor:
    """An uninitialised buffer like t, page-locked when t is a CPU tensor."""
    if t.is_cuda:
        return torch.empty_like(t)
    return torch.empty(t.shape, dtype=t.dtype, pin_memory=True)


def _code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return ICE_BF16
    if dtype == torch.float32:
        return ICE_F32
    raise ValueError(f"unsupported dtype {dtype}")


class IceIndex:
    """Owner of one ice_index handle (all units of a batch x layers x KV heads grid)."""

    def __init__(self, handle: int, params: ice_params, dtype: torch.dtype):
        self._h = ctypes.c_void_p(handle)
        self.params = params
        self.dtype = dtype

    # -- the four calls ------------------------------------------------------------
    @classmethod
    def build(cls, keys: torch.Tensor, values: torch.Tensor, *, page_size: int, n_q_heads: int,
              n_composite: int = 2, n_proj: int = 8, n_cand: int = 0, max_tokens: int | None = None,
              seed: int = 0, kv_host: bool = False, dir_kind: int = 0, stream=None) -> "IceIndex":
        """ice_build over keys/values shaped [batch, layers, kv_heads, n, d].

        kv_host places the page pool in pinned host memory (ICE_KV_HOST)."""
        if keys.dim() != 5 or keys.shape != values.shape:
            raise ValueError("keys/values must be [batch, layers, kv_heads, n, d] and equal in shape")
        B, Ly, H, n, d = keys.shape
        p = ice_params(d=d, n_kv_heads=H, n_q_heads=n_q_heads, n_layers=Ly, batch=B,
                       page_size=page_size, n_proj=n_proj, n_composite=n_composite, n_cand=n_cand,
                       dtype=_code(keys.dtype), max_tokens=n if max_tokens is None else max_tokens,
                       seed=seed, kv_location=KV_HOST if kv_host else KV_DEVICE, dir_kind=dir_kind)
        h = ctypes.c_void_p()
        kp = _dev_ptr(keys, values.dtype, "keys", host_ok=False) if n else 0
        vp = _dev_ptr(values, keys.dtype, "values", host_ok=False) if n else 0
        _check(_lib.ice_build(ctypes.byref(p), kp, vp, n, _stream(stream), ctypes.byref(h)),
               "ice_build")
        return cls(h.value, p, keys.dtype)

    def insert(self, k: torch.Tensor, v: torch.Tensor, stream=None):
        """ice_insert of one token per unit, k/v shaped [batch, layers, kv_heads, d]."""
        _check(_lib.ice_insert(self._h, _dev_ptr(k, self.dtype, "k"), _dev_ptr(v, self.dtype, "v"),
                               _stream(stream)), "ice_insert")

    def select(self, q: torch.Tensor, token_budget: int, page_ids: torch.Tensor | None = None,
               n_pages: torch.Tensor | None = None, stats: torch.Tensor | None = None, stream=None):
        """ice_select; returns (page_ids [units, n_sel] int32, n_pages [units] int32)."""
        U = self.n_units
        n_sel = token_budget // self.params.page_size
        dev = q.device if q.is_cuda else torch.device("cuda")  # q may be page-locked host memory
        if page_ids is None:
            page_ids = torch.empty((U, n_sel), dtype=torch.int32, device=dev)
        if n_pages is None:
            n_pages = torch.empty((U,), dtype=torch.int32, device=dev)
        sp = _dev_ptr(stats, torch.int32, "stats") if stats is not None else None
        _check(_lib.ice_select(self._h, _dev_ptr(q, self.dtype, "q"), int(token_budget),
                               _dev_ptr(page_ids, torch.int32, "page_ids"),
                               _dev_ptr(n_pages, torch.int32, "n_pages"), sp, _stream(stream)),
               "ice_select")
        return page_ids, n_pages

    def select_attn(self, q: torch.Tensor, token_budget: int, out: torch.Tensor | None = None,
                    page_ids: torch.Tensor | None = None, n_pages: torch.Tensor | None = None,
                    stats: torch.Tensor | None = None, stream=None):
        """ice_select_attn; returns (out, page_ids, n_pages)."""
        U = self.n_units
        n_sel = token_budget // self.params.page_size
        dev = q.device if q.is_cuda else torch.device("cuda")  # q may be page-locked host memory
        if page_ids is None:
            page_ids = torch.empty((U, n_sel), dtype=torch.int32, device=dev)
        if n_pages is None:
            n_pages = torch.empty((U,), dtype=torch.int32, device=dev)
        if out is None:
            out = _like(q)
        sp = _dev_ptr(stats, torch.int32, "stats") if stats is not None else None
        _check(_lib.ice_select_attn(self._h, _dev_ptr(q, self.dtype, "q"), int(token_budget),
                                    _dev_ptr(page_ids, torch.int32, "page_ids"),
                                    _dev_ptr(n_pages, torch.int32, "n_pages"), sp,
                                    _dev_ptr(out, self.dtype, "out"), _stream(stream)),
               "ice_select_attn")
        return out, page_ids, n_pages

    def select_attn_reuse(self, q: torch.Tensor, token_budget: int, r: int, page_ids: torch.Tensor,
                          n_pages: torch.Tensor, out: torch.Tensor | None = None,
                          reselected: torch.Tensor | None = None, stream=None):
        """ice_select_attn_reuse; page_ids/n_pages carry the selection between calls
        (pass the same tensors every step). Returns (out, page_ids, n_pages)."""
        if out is None:
            out = _like(q)
        _check(_lib.ice_select_attn_reuse(self._h, _dev_ptr(q, self.dtype, "q"), int(token_budget),
                                          int(r), _dev_ptr(page_ids, torch.int32, "page_ids"),
                                          _dev_ptr(n_pages, torch.int32, "n_pages"),
                                          (_dev_ptr(reselected, torch.int32, "reselected")
                                           if reselected is not None else None),
                                          _dev_ptr(out, self.dtype, "out"), _stream(stream)),
               "ice_select_attn_reuse")
        return out, page_ids, n_pages

    def debug_set_flags(self, flags: int):
        """ice_debug_set_flags (tests only): DEBUG_STALL_ATTN forces the fused call's
        bounded wait to run out."""
        _check(_lib.ice_debug_set_flags(self._h, int(flags)), "ice_debug_set_flags")

    def set_cluster_size(self, k: int):
        """ice_set_cluster_size: blocks per unit of the selection (0 automatic, 1, 2,
        4, 8 or 16)."""
        _check(_lib.ice_set_cluster_size(self._h, int(k)), "ice_set_cluster_size")

    def decode_step(self, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, token_budget: int,
                    page_ids: torch.Tensor, n_pages: torch.Tensor, out: torch.Tensor, stream=None):
        """ice_decode_step: insert (k, v) into every unit, then select + attend for q.
        Capturable in a CUDA graph (all buffers preallocated by the caller)."""
        _check(_lib.ice_decode_step(self._h, _dev_ptr(k, self.dtype, "k"), _dev_ptr(v, self.dtype, "v"),
                                    _dev_ptr(q, self.dtype, "q"), int(token_budget),
                                    _dev_ptr(page_ids, torch.int32, "page_ids"),
                                    _dev_ptr(n_pages, torch.int32, "n_pages"),
                                    _dev_ptr(out, self.dtype, "out"), _stream(stream)),
               "ice_decode_step")
        return out

    def select_heads(self, q: torch.Tensor, token_budget: int, stream=None):
        """ice_select_heads; returns (page_ids [units, G*n_sel] union, n_pages [units],
        head_page_ids [units, G, n_sel], head_n_pages [units, G])."""
        U, G = self.n_units, self.params.n_q_heads // self.params.n_kv_heads
        n_sel = token_budget // self.params.page_size
        dev = q.device if q.is_cuda else torch.device("cuda")
        hid = torch.empty((U, G, n_sel), dtype=torch.int32, device=dev)
        hn = torch.empty((U, G), dtype=torch.int32, device=dev)
        ids = torch.empty((U, G * n_sel), dtype=torch.int32, device=dev)
        n = torch.empty((U,), dtype=torch.int32, device=dev)
        _check(_lib.ice_select_heads(self._h, _dev_ptr(q, self.dtype, "q"), int(token_budget),
                                     hid.data_ptr(), hn.data_ptr(), ids.data_ptr(), n.data_ptr(),
                                     _stream(stream)), "ice_select_heads")
        return ids, n, hid, hn

    def reuse_reset(self, stream=None):
        _check(_lib.ice_reuse_reset(self._h, _stream(stream)), "ice_reuse_reset")

    def sparse_attn(self, q: torch.Tensor, page_ids: torch.Tensor, n_pages: torch.Tensor,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """ice_sparse_attn; returns out shaped like q."""
        if out is None:
            out = _like(q)
        _check(_lib.ice_sparse_attn(self._h, _dev_ptr(q, self.dtype, "q"),
                                    _dev_ptr(page_ids, torch.int32, "page_ids"),
                                    _dev_ptr(n_pages, torch.int32, "n_pages"),
                                    int(page_ids.shape[-1]), _dev_ptr(out, self.dtype, "out"),
                                    _stream(stream)), "ice_sparse_attn")
        return out

    # -- status, info, teardown ---------------------------------------------------------
    def get_error(self, stream=None) -> int:
        return int(_lib.ice_get_error(self._h, _stream(stream)))

    def check(self, stream=None):
        _check(self.get_error(stream), "device status")

    def info(self) -> ice_info:
        inf = ice_info()
        _check(_lib.ice_get_info(self._h, ctypes.byref(inf)), "ice_get_info")
        return inf

    @property
    def n_units(self) -> int:
        p = self.params
        return p.batch * p.n_layers * p.n_kv_heads

    def destroy(self):
        if self._h and self._h.value:
            _lib.ice_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    # -- debug views --------------------------------------------------------------------
    def dump(self, unit: int, stream=None) -> dict:
        """Decoded ice_debug_dump of one unit (see include/ice.h for the layout)."""
        need = int(_lib.ice_debug_dump(self._h, unit, None, 0, _stream(stream)))
        if need < 0:
            raise IceError(need, "ice_debug_dump")
        buf = np.zeros(need, dtype=np.uint8)
        _check(int(_lib.ice_debug_dump(self._h, unit, buf.ctypes.data, need, _stream(stream))),
               "ice_debug_dump")
        hdr = buf[:128].view(np.int64)
        L, P, C, n, e = (int(x) for x in hdr[:5])
        out = {"L": L, "P": P, "C": C, "n": n, "e": e, "n_leaf": hdr[5:5 + L].tolist(),
               "next_id": hdr[9:9 + L].tolist(), "comp": []}
        o = 128
        for _ in range(L):
            lk = buf[o:o + C * 16].view(np.uint32).reshape(C, 4)
            o += C * 16
            rec = buf[o:o + C * 16].reshape(C, 16)
            o += C * 16
            meta = rec[:, 8:12].copy().view(np.uint32).reshape(C)
            lo = rec[:, :8].astype(np.int32)
            t = lk[:, 3].astype(np.int32)
            # known bits of code j at prefix length t (Morton order, code j at bit j of each byte)
            jj = np.arange(8)[None, :]
            bj = np.where(t[:, None] >= 64, 8, np.clip((t[:, None] + 7 - jj) >> 3, 0, 8))
            hi = lo | ((1 << (8 - bj)) - 1)
            rec_t = rec[:, 12:16].copy().view(np.uint32).reshape(C).astype(np.int32)
            cnt = buf[o:o + C * 4].view(np.int32)
            o += C * 4
            stok = buf[o:o + C * P * 4].view(np.int32).reshape(C, P)
            o += C * P * 4
            skey = buf[o:o + C * P * 8].view(np.uint64).reshape(C, P)
            o += C * P * 8
            pm = lk[:, 0].astype(np.uint64) | (lk[:, 1].astype(np.uint64) << np.uint64(32))
            out["comp"].append({"pm": pm, "pt": lk[:, 2].copy(), "t": t, "rec_t": rec_t,
                                "lo": lo, "hi": hi,
                                "id": (meta >> 8).astype(np.int32), "cnt": (meta & 0xFF).astype(np.int32),
                                "list_cnt": cnt.copy(), "slot_tok": stok.copy(), "slot_key": skey.copy()})
        mt = self.info().max_tokens
        out["tok_loc"] = buf[o:o + 4 * mt].view(np.int32).copy()
        o += 4 * mt
        if L > 1:
            out["slot_loc1"] = buf[o:o + C * P * 4].view(np.int32).reshape(C, P).copy()
            o += C * P * 4
            out["tok_slot1"] = buf[o:o + 4 * mt].view(np.int32).copy()
        return out

    def page(self, unit: int, page_id: int, stream=None):
        """K and V rows of one page as torch CPU tensors [P, d]."""
        P, d = self.params.page_size, self.params.d
        hk = torch.empty((P, d), dtype=self.dtype)
        hv = torch.empty((P, d), dtype=self.dtype)
        _check(_lib.ice_debug_page(self._h, unit, page_id, hk.data_ptr(), hv.data_ptr(),
                                   _stream(stream)), "ice_debug_page")
        return hk, hv


def key_codes_noalloc(keys: torch.Tensor, *, n_composite: int = 2, n_proj: int = 8, seed: int = 0,
                      morton_out: torch.Tensor | None = None, e_out: torch.Tensor | None = None,
                      stream=None):
    """ice_key_codes_noalloc on keys [batch, layers, kv_heads, n, d].

    Returns (morton [n_composite, units, n] as int64 bit patterns, e [units]).
    Pass preallocated outputs to keep the call free of allocations."""
    B, Ly, H, n, d = keys.shape
    U = B * Ly * H
    p = ice_params(d=d, n_kv_heads=H, n_q_heads=H, n_layers=Ly, batch=B, page_size=1,
                   n_proj=n_proj, n_composite=n_composite, n_cand=0, dtype=_code(keys.dtype),
                   max_tokens=n, seed=seed)
    if morton_out is None:
        morton_out = torch.empty((n_composite, U, n), dtype=torch.int64, device=keys.device)
    if e_out is None:
        e_out = torch.empty((U,), dtype=torch.int32, device=keys.device)
    _check(_lib.ice_key_codes_noalloc(ctypes.byref(p), _dev_ptr(keys, None, "keys", host_ok=False), n,
                                      _dev_ptr(morton_out, torch.int64, "morton_out", host_ok=False),
                                      _dev_ptr(e_out, torch.int32, "e_out", host_ok=False),
                                      _stream(stream)),
           "ice_key_codes_noalloc")
    return morton_out, e_out


def raw_library() -> ctypes.CDLL:
    """The loaded libice.so (for tests that call the C ABI directly)."""
    return _lib

"""CPU oracle of differentiated KV compaction — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The product
path (``differentiated_kv_cache_gb300``) never does, and the two share no code.

The arithmetic lives in ``dkv_oracle.c`` (plain C, fp64 scores and attention,
pinned fp32 codec and thresholds); this module compiles it with gcc and wraps
it with ctypes and numpy.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

TIER_PRUNE, TIER_LO, TIER_HI, TIER_MID = 0, 1, 2, 3
ERR = dict(OK=0, ARG=-1, STATE=-3, NO_PAGES=-4, TABLE_FULL=-5, CHECK=-7)


def build(force: bool = False) -> str:
    """Compile the oracle (IEEE arithmetic, no contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                        "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_layers", "n_kv_heads", "group_size", "page_bytes",
                                          "n_pages", "max_requests", "max_seq_len", "t_hi", "t_lo",
                                          "lo_enabled")] + \
               [("alpha_h", C.c_float), ("alpha_l", C.c_float)] + \
               [(n, C.c_int32) for n in ("window", "grant_slack", "reclaim_in_decode", "mid_enabled")] + \
               [("alpha_m", C.c_float), ("t_mid", C.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # DKV_ORACLE_LIB: load a separately built copy instead (the test that
            # plants mistakes in copies of the oracle uses it)
            L = C.CDLL(os.environ.get("DKV_ORACLE_LIB") or build())
            P, I, I64 = C.c_void_p, C.c_int, C.c_int64
            L.orc_half_to_float.argtypes = [C.c_uint16]; L.orc_half_to_float.restype = C.c_float
            L.orc_float_to_half.argtypes = [C.c_float]; L.orc_float_to_half.restype = C.c_uint16
            L.orc_quantize.argtypes = [P, I, I, P, P, P]; L.orc_quantize.restype = None
            L.orc_dequant.argtypes = [C.c_uint16, C.c_uint16, I]; L.orc_dequant.restype = C.c_float
            L.orc_pool_new.argtypes = [P]; L.orc_pool_new.restype = P
            L.orc_pool_free.argtypes = [P]; L.orc_pool_free.restype = None
            L.orc_geometry.argtypes = [P, P]; L.orc_geometry.restype = None
            for f in ("orc_pages", "orc_list", "orc_pointers", "orc_table", "orc_head_counts",
                      "orc_req_state"):
                getattr(L, f).argtypes = [P]; getattr(L, f).restype = P
            L.orc_unit_scores.argtypes = [I, I, P, I64, P, I64, I64, P]; L.orc_unit_scores.restype = None
            L.orc_prompt_step.argtypes = [P, I, I, P, P, P, P, P, P, P]; L.orc_prompt_step.restype = I
            L.orc_decode_step.argtypes = [P, I, I, P, P, P]; L.orc_decode_step.restype = I
            L.orc_unit_attention.argtypes = [P, I, I, I, P, P, P]; L.orc_unit_attention.restype = I
            L.orc_decode_attention.argtypes = [P, I, I, P, P, P, I]; L.orc_decode_attention.restype = I
            L.orc_free_request.argtypes = [P, I]; L.orc_free_request.restype = I
            L.orc_set_thresholds.argtypes = [P, I, P, P]; L.orc_set_thresholds.restype = I
            L.orc_prefill_attention.argtypes = [I, I, P, I64, P, P, I64, P, P]
            L.orc_prefill_attention.restype = None
            L.orc_prefill_rows.argtypes = [I, I, P, P, I64, P, P, I64, P, P]
            L.orc_prefill_rows.restype = None
            L.orc_thresholds.argtypes = [P]; L.orc_thresholds.restype = P
            L.orc_set_mid_thresholds.argtypes = [P, I, P]; L.orc_set_mid_thresholds.restype = I
            L.orc_mid_thresholds.argtypes = [P]; L.orc_mid_thresholds.restype = P
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags.c_contiguous
    return a.ctypes.data_as(C.c_void_p)


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float16)).view(np.uint16)


# ---- codec ---------------------------------------------------------------
def float_to_half_bits(x: float) -> int:
    return int(lib().orc_float_to_half(C.c_float(x)))


def half_bits_to_float(h: int) -> float:
    return float(lib().orc_half_to_float(C.c_uint16(h)))


def quantize(x: np.ndarray, bits: int):
    """Quantize one fp32 vector: returns (codes uint8, scale fp16 bits, zero fp16 bits)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.size, dtype=np.uint8)
    s = C.c_uint16(); z = C.c_uint16()
    lib().orc_quantize(_ptr(x), x.size, bits, _ptr(codes), C.byref(s), C.byref(z))
    return codes, int(s.value), int(z.value)


def dequant(scale_bits: int, zero_bits: int, codes: np.ndarray) -> np.ndarray:
    L = lib()
    return np.array([L.orc_dequant(scale_bits, zero_bits, int(c)) for c in codes], dtype=np.float32)


def unit_scores(k_head: np.ndarray, q_group: np.ndarray) -> np.ndarray:
    """fp64 prompt scores S of one KV head. k_head: fp16 [N0, 128]; q_group:
    fp16 [32, G, 128] (row o = position N0-32+o)."""
    k = _u16(k_head); q = _u16(q_group)
    n0, G = k.shape[0], q.shape[1]
    S = np.zeros(n0, dtype=np.float64)
    lib().orc_unit_scores(n0, G, _ptr(k), 128, _ptr(q), G * 128, 128, _ptr(S))
    return S


def prefill_attention(q_group: np.ndarray, k_head: np.ndarray, v_head: np.ndarray):
    """fp64 causal attention of one KV head's G query heads over a prompt.
    q_group fp16 [N0, G, 128]; k_head, v_head fp16 [N0, 128]. Returns
    (out fp64 [N0, G, 128], lse2 fp64 [N0, G]: base-2 log-sum-exp of the
    scaled logits)."""
    q = _u16(q_group); k = _u16(k_head); v = _u16(v_head)
    n0, G = q.shape[0], q.shape[1]
    out = np.zeros((n0, G, 128), np.float64)
    lse2 = np.zeros((n0, G), np.float64)
    lib().orc_prefill_attention(n0, G, _ptr(q), G * 128, _ptr(k), _ptr(v), 128, _ptr(out), _ptr(lse2))
    return out, lse2


def prefill_rows(positions, q_rows: np.ndarray, k_head: np.ndarray, v_head: np.ndarray):
    """The same attention at selected positions only: q_rows fp16 [m, G, 128]
    (row r is the query at positions[r]); k_head, v_head fp16 [n, 128] with
    n > max(positions). Returns (out fp64 [m, G, 128], lse2 fp64 [m, G])."""
    pos = np.ascontiguousarray(positions, dtype=np.int32).reshape(-1)
    q = _u16(q_rows); k = _u16(k_head); v = _u16(v_head)
    m, G = q.shape[0], q.shape[1]
    assert pos.size == m and (pos >= 0).all() and int(pos.max()) < k.shape[0]
    out = np.zeros((m, G, 128), np.float64)
    lse2 = np.zeros((m, G), np.float64)
    lib().orc_prefill_rows(m, G, _ptr(pos), _ptr(q), G * 128, _ptr(k), _ptr(v), 128, _ptr(out), _ptr(lse2))
    return out, lse2


# ---- pool -------------------------------------------------------------------
class Pool:
    """The oracle's pool: pages, free list, pointers, bidirectional table,
    per-head counters and per-request state, as plain host arrays."""

    def __init__(self, cfg: dict):
        self.cfg = dict(cfg)
        c = _Config(n_layers=cfg["n_layers"], n_kv_heads=cfg["n_kv_heads"], group_size=cfg["group_size"],
                    page_bytes=cfg["page_bytes"], n_pages=cfg["n_pages"], max_requests=cfg["max_requests"],
                    max_seq_len=cfg["max_seq_len"], t_hi=cfg.get("tokens_per_hi_page", 0),
                    t_lo=cfg.get("tokens_per_lo_page", 0), lo_enabled=cfg["lo_enabled"],
                    alpha_h=cfg["alpha_h"], alpha_l=cfg["alpha_l"], window=cfg["recent_window"],
                    grant_slack=cfg["prompt_grant_slack"], reclaim_in_decode=cfg["reclaim_in_decode"],
                    mid_enabled=cfg.get("mid_enabled", 0), alpha_m=cfg.get("alpha_m", 0.0),
                    t_mid=cfg.get("tokens_per_mid_page", 0))
        self.mid = bool(cfg.get("mid_enabled", 0))
        self._h = lib().orc_pool_new(C.byref(c))
        g = np.zeros(28, dtype=np.int32)
        lib().orc_geometry(self._h, _ptr(g))
        self.t_hi, self.t_lo, self.table_len = int(g[0]), int(g[1]), int(g[2])
        self.hi_off, self.lo_off = g[3:9].copy(), g[9:15].copy()
        self.hi_used, self.lo_used = int(g[15]), int(g[16])
        # the third level (mid, K8V2) and the one-way part of the table rows
        self.t_mid, self.mid_len = int(g[17]), int(g[18])
        self.mid_off, self.mid_used = g[19:25].copy(), int(g[25])
        self.row_len, self.cstride = int(g[26]), int(g[27])

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_pool_free(self._h)
            self._h = None

    def _view(self, fn, dtype, count):
        addr = getattr(lib(), fn)(self._h)
        return np.ctypeslib.as_array(C.cast(addr, C.POINTER(np.ctypeslib.as_ctypes_type(dtype))),
                                     shape=(count,))

    # live views of the state ----------------------------------------------------
    @property
    def pages(self):
        c = self.cfg
        return self._view("orc_pages", np.uint8, c["n_pages"] * c["page_bytes"]).reshape(c["n_pages"], c["page_bytes"])

    @property
    def free_list(self):
        return self._view("orc_list", np.int32, self.cfg["n_pages"])

    @property
    def pointers(self):
        return self._view("orc_pointers", np.int64, 2)

    @property
    def table(self):
        c = self.cfg
        n = c["n_layers"] * c["max_requests"] * c["n_kv_heads"]
        return self._view("orc_table", np.int32, n * self.row_len).reshape(
            c["n_layers"], c["max_requests"], c["n_kv_heads"], self.row_len)

    @property
    def head_counts(self):
        c = self.cfg
        n = c["n_layers"] * c["max_requests"] * c["n_kv_heads"]
        return self._view("orc_head_counts", np.int32, n * self.cstride).reshape(
            c["n_layers"], c["max_requests"], c["n_kv_heads"], self.cstride)

    @property
    def req_state(self):
        c = self.cfg
        return self._view("orc_req_state", np.int32, c["n_layers"] * c["max_requests"] * 4).reshape(
            c["n_layers"], c["max_requests"], 4)

    # operations -------------------------------------------------------------------
    def prompt(self, layer, slots, lens, k, v, q_obs=None, scores_in=None, want_scores=False):
        slots = np.ascontiguousarray(slots, dtype=np.int32)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        ku, vu = _u16(k), _u16(v)
        qu = None if q_obs is None else _u16(q_obs)
        si = None if scores_in is None else np.ascontiguousarray(scores_in, dtype=np.float32)
        so = np.zeros((int(lens.sum()), self.cfg["n_kv_heads"]), np.float32) if want_scores else None
        rc = lib().orc_prompt_step(self._h, layer, len(slots), _ptr(slots), _ptr(lens), _ptr(ku),
                                   _ptr(vu), _ptr(qu), _ptr(si), _ptr(so))
        return (rc, so) if want_scores else rc

    def decode(self, layer, slots, k, v):
        slots = np.ascontiguousarray(slots, dtype=np.int32)
        return lib().orc_decode_step(self._h, layer, len(slots), _ptr(slots), _ptr(_u16(k)), _ptr(_u16(v)))

    def attention(self, layer, slots, q, update_scores=False):
        slots = np.ascontiguousarray(slots, dtype=np.int32)
        qu = _u16(q)
        out = np.zeros(qu.shape, dtype=np.float64)
        rc = lib().orc_decode_attention(self._h, layer, len(slots), _ptr(slots), _ptr(qu), _ptr(out),
                                        int(bool(update_scores)))
        return rc, out

    def unit_attention(self, layer, slot, kvh, q_group):
        """fp64 attention of one KV head (q_group fp16 [G, 128]); returns
        (out [G,128] fp64, pmax over stored tokens (hi slots, mid slots, then
        lo slots))."""
        qu = _u16(q_group)
        cnt = self.head_counts[layer, slot, kvh]
        n = int(cnt[0] + cnt[1] + (cnt[4] if self.mid else 0))
        out = np.zeros(qu.shape, np.float64)
        pm = np.zeros(max(n, 1), np.float64)
        lib().orc_unit_attention(self._h, layer, slot, kvh, _ptr(qu), _ptr(out), _ptr(pm))
        return out, pm[:n]

    def free_request(self, slot):
        return lib().orc_free_request(self._h, int(slot))

    def set_thresholds(self, layer, alpha_h, alpha_l):
        """Per-head thresholds of one layer (arrays of n_kv_heads floats)."""
        ah = np.ascontiguousarray(alpha_h, dtype=np.float32)
        al = np.ascontiguousarray(alpha_l, dtype=np.float32)
        assert ah.size == al.size == self.cfg["n_kv_heads"]
        return lib().orc_set_thresholds(self._h, int(layer), _ptr(ah), _ptr(al))

    def set_mid_thresholds(self, layer, alpha_m):
        """Per-head thresholds of the mid level of one layer (n_kv_heads floats)."""
        am = np.ascontiguousarray(alpha_m, dtype=np.float32)
        assert am.size == self.cfg["n_kv_heads"]
        return lib().orc_set_mid_thresholds(self._h, int(layer), _ptr(am))

    @property
    def mid_thresholds(self):
        """Live view [layer][kvh] of alpha_m."""
        c = self.cfg
        return self._view("orc_mid_thresholds", np.float32, c["n_layers"] * c["n_kv_heads"]).reshape(
            c["n_layers"], c["n_kv_heads"])

    @property
    def thresholds(self):
        """Live view [layer][kvh][alpha_h, alpha_l]."""
        c = self.cfg
        return self._view("orc_thresholds", np.float32, c["n_layers"] * c["n_kv_heads"] * 2).reshape(
            c["n_layers"], c["n_kv_heads"], 2)

    def snapshot(self) -> dict:
        return dict(pages=self.pages.copy(), free_list=self.free_list.copy(),
                    pointers=self.pointers.copy(), table=self.table.copy(),
                    head_counts=self.head_counts.copy(), req_state=self.req_state.copy(),
                    thresholds=self.thresholds.copy(), mid_thresholds=self.mid_thresholds.copy())

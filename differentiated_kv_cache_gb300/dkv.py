"""ctypes binding of libdkv (include/dkv.h): same entry-point names, argument
marshalling only. Every step of the compaction and attention path runs in the
library's CUDA kernels; there is no fallback — importing this module on a
machine without the built library raises.

Tensors are PyTorch CUDA tensors (device memory and streams only); host
arrays are anything numpy can turn into int32.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

DKV_OK, DKV_ERR_ARG, DKV_ERR_CUDA, DKV_ERR_STATE = 0, -1, -2, -3
DKV_ERR_NO_PAGES, DKV_ERR_TABLE_FULL, DKV_ERR_TIMEOUT, DKV_ERR_CHECK, DKV_ERR_UNSUPPORTED = -4, -5, -6, -7, -8
DKV_ERR_SCRATCH = -9
DKV_ATTN_STATIC_SCRATCH_BYTES = 64 << 20
DKV_PROMPT, DKV_DECODE = 0, 1

EXPORTED = ("dkv_pool_create", "dkv_pool_destroy", "dkv_pool_geometry", "dkv_compact_step",
            "dkv_decode_attention", "dkv_decode_attention_static", "dkv_free_request", "dkv_pool_status", "dkv_pool_clear_error",
            "dkv_pool_export", "dkv_pool_set_thresholds", "dkv_pool_set_mid_thresholds", "dkv_prefill_attention",
            "dkv_compact_step_prefilled", "dkv_strerror")


class dkv_config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "n_layers", "n_kv_heads", "group_size", "head_dim", "page_bytes", "n_pages", "max_requests",
        "max_seq_len", "tokens_per_hi_page", "tokens_per_lo_page", "lo_enabled")] + \
        [("alpha_h", C.c_float), ("alpha_l", C.c_float)] + \
        [(n, C.c_int32) for n in ("recent_window", "obs_window", "prompt_grant_slack", "reclaim_in_decode",
                                  "mid_enabled")] + \
        [("alpha_m", C.c_float), ("tokens_per_mid_page", C.c_int32)]


class dkv_geometry(C.Structure):
    _fields_ = [("t_hi", C.c_int32), ("t_lo", C.c_int32), ("table_len", C.c_int32),
                ("hi_off", C.c_int32 * 6), ("lo_off", C.c_int32 * 6), ("hi_used", C.c_int32),
                ("lo_used", C.c_int32), ("t_mid", C.c_int32), ("mid_table_len", C.c_int32),
                ("row_len", C.c_int32), ("count_stride", C.c_int32), ("mid_off", C.c_int32 * 6),
                ("mid_used", C.c_int32)]


class dkv_status(C.Structure):
    _fields_ = [("error", C.c_int32), ("error_info", C.c_int32)] + \
        [(n, C.c_int64) for n in ("list_start", "list_end", "free_pages", "hi_tokens", "lo_tokens",
                                  "hi_pages", "lo_pages", "mid_tokens", "mid_pages")]


class dkv_snapshot(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("pages", "free_list", "table", "head_counts", "req_state",
                                          "pointers")]


class DkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {dkv_strerror(code)} ({code})")
        self.code = code


_lib = None


def lib_path() -> str:
    return _build.LIB


def load() -> C.CDLL:
    """Load libdkv.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libdkv is not built ({_build.LIB}); run __graft_entry__.build()")
        L = C.CDLL(_build.LIB)
        P, I = C.c_void_p, C.c_int32
        L.dkv_pool_create.argtypes = [C.POINTER(dkv_config), C.c_int, C.POINTER(C.c_void_p)]
        L.dkv_pool_destroy.argtypes = [P]
        L.dkv_pool_geometry.argtypes = [P, C.POINTER(dkv_geometry)]
        L.dkv_compact_step.argtypes = [P, I, I, I, P, P, P, P, P, P, P, P]
        L.dkv_decode_attention.argtypes = [P, I, I, P, P, P, I, P]
        L.dkv_prefill_attention.argtypes = [P, I, P, P, P, P, P, P, P]
        L.dkv_compact_step_prefilled.argtypes = [P, I, I, P, P, P, P, P, P, P, P]
        L.dkv_free_request.argtypes = [P, I, P]
        L.dkv_pool_set_thresholds.argtypes = [P, I, P, P, P]
        L.dkv_pool_set_mid_thresholds.argtypes = [P, I, P, P]
        L.dkv_pool_status.argtypes = [P, C.POINTER(dkv_status)]
        L.dkv_pool_clear_error.argtypes = [P]
        L.dkv_pool_export.argtypes = [P, C.POINTER(dkv_snapshot)]
        L.dkv_strerror.argtypes = [C.c_int]
        L.dkv_strerror.restype = C.c_char_p
        for f in EXPORTED:
            if f != "dkv_strerror":
                getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def dkv_strerror(code: int) -> str:
    return load().dkv_strerror(int(code)).decode()


def _check(rc: int, what: str) -> int:
    if rc != DKV_OK:
        raise DkvError(rc, what)
    return rc


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))


def _dptr(t, dtype=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def make_config(**kw) -> dkv_config:
    c = dkv_config()
    defaults = dict(head_dim=128, page_bytes=4096, tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=1,
                    alpha_h=2.0, alpha_l=0.25, recent_window=64, obs_window=32, prompt_grant_slack=1,
                    reclaim_in_decode=1, mid_enabled=0, alpha_m=0.0, tokens_per_mid_page=0)
    defaults.update(kw)
    for name, _ in dkv_config._fields_:
        setattr(c, name, defaults[name])
    return c


def dkv_pool_create(cfg, device: int = 0) -> C.c_void_p:
    if isinstance(cfg, dict):
        cfg = make_config(**cfg)
    h = C.c_void_p()
    _check(load().dkv_pool_create(C.byref(cfg), int(device), C.byref(h)), "dkv_pool_create")
    return h


def dkv_pool_destroy(pool) -> None:
    _check(load().dkv_pool_destroy(pool), "dkv_pool_destroy")


def dkv_pool_geometry(pool) -> dict:
    g = dkv_geometry()
    _check(load().dkv_pool_geometry(pool, C.byref(g)), "dkv_pool_geometry")
    return dict(t_hi=g.t_hi, t_lo=g.t_lo, table_len=g.table_len, hi_off=list(g.hi_off), lo_off=list(g.lo_off),
                hi_used=g.hi_used, lo_used=g.lo_used, t_mid=g.t_mid, mid_table_len=g.mid_table_len,
                row_len=g.row_len, count_stride=g.count_stride, mid_off=list(g.mid_off), mid_used=g.mid_used)


def dkv_compact_step(pool, layer: int, mode: int, req_slots, seq_lens, k, v, q_obs=None, scores_in=None,
                     scores_out=None, stream=None, check: bool = True) -> int:
    import torch
    slots = _i32(req_slots)
    lens = None if seq_lens is None else _i32(seq_lens)
    rc = load().dkv_compact_step(
        pool, int(layer), int(mode), int(slots.size), slots.ctypes.data,
        None if lens is None else lens.ctypes.data,
        _dptr(k, torch.float16, "k"), _dptr(v, torch.float16, "v"), _dptr(q_obs, torch.float16, "q_obs"),
        _dptr(scores_in, torch.float32, "scores_in"), _dptr(scores_out, torch.float32, "scores_out"),
        _stream(stream))
    return _check(rc, "dkv_compact_step") if check else rc


def dkv_prefill_attention(pool, seq_lens, q, k, v, out, lse_obs=None, stream=None, check: bool = True) -> int:
    """Causal attention over whole prompts (requests back to back): q fp16
    [sum(seq_lens)][Hq][128], k and v fp16 [sum(seq_lens)][Hkv][128], out fp32
    like q; lse_obs None or fp32 [n_req][Hq][32] for the last 32 rows'
    base-2 log-sum-exps."""
    import torch
    lens = _i32(seq_lens)
    rc = load().dkv_prefill_attention(pool, int(lens.size), lens.ctypes.data,
                                      _dptr(q, torch.float16, "q"), _dptr(k, torch.float16, "k"),
                                      _dptr(v, torch.float16, "v"), _dptr(out, torch.float32, "out"),
                                      _dptr(lse_obs, torch.float32, "lse_obs"), _stream(stream))
    return _check(rc, "dkv_prefill_attention") if check else rc


def dkv_compact_step_prefilled(pool, layer: int, req_slots, seq_lens, k, v, q_obs, lse_obs, scores_out=None,
                               stream=None, check: bool = True) -> int:
    """PROMPT compaction with the observation rows' log-sum-exps given by
    dkv_prefill_attention."""
    import torch
    slots = _i32(req_slots)
    lens = _i32(seq_lens)
    rc = load().dkv_compact_step_prefilled(
        pool, int(layer), int(slots.size), slots.ctypes.data, lens.ctypes.data,
        _dptr(k, torch.float16, "k"), _dptr(v, torch.float16, "v"), _dptr(q_obs, torch.float16, "q_obs"),
        _dptr(lse_obs, torch.float32, "lse_obs"), _dptr(scores_out, torch.float32, "scores_out"), _stream(stream))
    return _check(rc, "dkv_compact_step_prefilled") if check else rc


def dkv_decode_attention(pool, layer: int, req_slots, q, out, update_scores: bool = False, stream=None,
                         check: bool = True) -> int:
    import torch
    slots = _i32(req_slots)
    rc = load().dkv_decode_attention(pool, int(layer), int(slots.size), slots.ctypes.data,
                                     _dptr(q, torch.float16, "q"), _dptr(out, torch.float32, "out"),
                                     int(bool(update_scores)), _stream(stream))
    return _check(rc, "dkv_decode_attention") if check else rc


def dkv_decode_attention_static(pool, layer: int, req_slots, q, out, update_scores: bool = False, stream=None,
                                check: bool = True) -> int:
    """dkv_decode_attention working in the library's fixed 64 MiB device
    array instead of the pool's scratch (for callers that cannot allocate
    device memory). Calls that overlap on the GPU race on the array."""
    import torch
    slots = _i32(req_slots)
    rc = load().dkv_decode_attention_static(pool, int(layer), int(slots.size), slots.ctypes.data,
                                            _dptr(q, torch.float16, "q"), _dptr(out, torch.float32, "out"),
                                            int(bool(update_scores)), _stream(stream))
    return _check(rc, "dkv_decode_attention_static") if check else rc


def dkv_pool_set_thresholds(pool, layer: int, alpha_h, alpha_l, stream=None, check: bool = True) -> int:
    """Per-KV-head thresholds of one layer (host arrays of n_kv_heads floats)."""
    ah = np.ascontiguousarray(alpha_h, dtype=np.float32)
    al = np.ascontiguousarray(alpha_l, dtype=np.float32)
    rc = load().dkv_pool_set_thresholds(pool, int(layer), ah.ctypes.data,
                                        al.ctypes.data, _stream(stream))
    return _check(rc, "dkv_pool_set_thresholds") if check else rc


def dkv_pool_set_mid_thresholds(pool, layer: int, alpha_m, stream=None, check: bool = True) -> int:
    """Per-KV-head thresholds of the mid tier of one layer (n_kv_heads floats)."""
    am = np.ascontiguousarray(alpha_m, dtype=np.float32)
    rc = load().dkv_pool_set_mid_thresholds(pool, int(layer), am.ctypes.data, _stream(stream))
    return _check(rc, "dkv_pool_set_mid_thresholds") if check else rc


def dkv_free_request(pool, req_slot: int, stream=None, check: bool = True) -> int:
    rc = load().dkv_free_request(pool, int(req_slot), _stream(stream))
    return _check(rc, "dkv_free_request") if check else rc


def dkv_pool_status(pool) -> dict:
    s = dkv_status()
    _check(load().dkv_pool_status(pool, C.byref(s)), "dkv_pool_status")
    return {n: getattr(s, n) for n, _ in dkv_status._fields_}


def dkv_pool_clear_error(pool) -> None:
    _check(load().dkv_pool_clear_error(pool), "dkv_pool_clear_error")


def dkv_pool_export(pool, cfg: dict, table_len: int, pages: bool = True, count_stride: int = 4) -> dict:
    """Host copy of the device state as numpy arrays, shaped like the oracle's
    (table_len: entries of a table row, the geometry's row_len; count_stride:
    ints of a head's counters, 8 with the mid tier)."""
    nl, mr, hk, npg = cfg["n_layers"], cfg["max_requests"], cfg["n_kv_heads"], cfg["n_pages"]
    out = dict(
        pages=np.zeros((npg, cfg["page_bytes"]) if pages else (0,), np.uint8),
        free_list=np.zeros(npg, np.int32),
        table=np.zeros((nl, mr, hk, table_len), np.int32),
        head_counts=np.zeros((nl, mr, hk, count_stride), np.int32),
        req_state=np.zeros((nl, mr, 4), np.int32),
        pointers=np.zeros(2, np.int64))
    snap = dkv_snapshot()
    for name in ("free_list", "table", "head_counts", "req_state", "pointers"):
        setattr(snap, name, out[name].ctypes.data)
    snap.pages = out["pages"].ctypes.data if pages else None
    _check(load().dkv_pool_export(pool, C.byref(snap)), "dkv_pool_export")
    return out

"""Small helpers shared by the GPU tests: a pool wrapper over the C-ABI
binding and vectorised readers of a snapshot's stored positions and scores."""
from __future__ import annotations

import numpy as np

import differentiated_kv_cache_gb300 as dkv
from tests import pagefmt


class GPool:
    def __init__(self, cfg: dict):
        import torch
        self.torch = torch
        self.cfg = dict(cfg)
        self.h = dkv.dkv_pool_create(dkv.make_config(**{k: v for k, v in cfg.items()
                                                         if k in dict(dkv.dkv_config._fields_)}), 0)
        self.geom = dkv.dkv_pool_geometry(self.h)
        self.t_hi, self.t_lo, self.table_len = self.geom["t_hi"], self.geom["t_lo"], self.geom["table_len"]
        # three-tier pools: rows of row_len entries (two-way part, then the
        # one-way mid part), counters of 8 ints
        self.t_mid, self.row_len, self.cstride = self.geom["t_mid"], self.geom["row_len"], self.geom["count_stride"]

    def close(self):
        if self.h is not None:
            dkv.dkv_pool_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def dev(self, a, dtype=None):
        t = self.torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            t = t.to(dtype)
        return t.cuda()

    def prompt(self, layer, slots, lens, k, v, q_obs=None, scores_in=None, want_scores=False, check=True):
        torch = self.torch
        kd, vd = self.dev(k), self.dev(v)
        qd = None if q_obs is None else self.dev(q_obs)
        si = None if scores_in is None else self.dev(scores_in.astype(np.float32))
        so = torch.zeros((int(np.sum(lens)), self.cfg["n_kv_heads"]), dtype=torch.float32,
                         device="cuda") if want_scores else None
        rc = dkv.dkv_compact_step(self.h, layer, dkv.DKV_PROMPT, slots, lens, kd, vd, qd, si, so, check=check)
        torch.cuda.synchronize()
        return (rc, so.cpu().numpy()) if want_scores else rc

    def decode(self, layer, slots, k, v, check=True):
        rc = dkv.dkv_compact_step(self.h, layer, dkv.DKV_DECODE, slots, None, self.dev(k), self.dev(v),
                                  check=check)
        self.torch.cuda.synchronize()
        return rc

    def attention(self, layer, slots, q, update=False):
        torch = self.torch
        qd = self.dev(q)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        dkv.dkv_decode_attention(self.h, layer, slots, qd, out, update)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def free(self, slot, check=True):
        rc = dkv.dkv_free_request(self.h, slot, check=check)
        self.torch.cuda.synchronize()
        return rc

    def snapshot(self, pages=True):
        return dkv.dkv_pool_export(self.h, self.cfg, self.row_len, pages=pages, count_stride=self.cstride)

    def status(self):
        return dkv.dkv_pool_status(self.h)


def stored(snap: dict, head: tuple, t_hi: int, t_lo: int, seg: int, dtype) -> tuple[np.ndarray, np.ndarray]:
    """(hi values, lo values) of segment `seg` (4 = score, 5 = position) of a
    head's stored slots, in slot order."""
    cnt = snap["head_counts"][head]
    row = snap["table"][head]
    L = row.shape[0]
    out = []
    for tier, n, t in ((pagefmt.HI, int(cnt[0]), t_hi), (pagefmt.LO, int(cnt[1]), t_lo)):
        kb, vb = pagefmt.BITS[tier]
        offs, _ = pagefmt.segment_offsets(t, kb, vb)
        vals = []
        for x in range(-(-n // t)):
            page = row[x] if tier == pagefmt.HI else row[L - 1 - x]
            nv = min(t, n - x * t)
            vals.append(snap["pages"][page, offs[seg]: offs[seg] + 4 * nv].view(dtype))
        out.append(np.concatenate(vals) if vals else np.zeros(0, dtype))
    return out[0], out[1]


def tiers_of(snap: dict, head: tuple, n: int, t_hi: int, t_lo: int) -> np.ndarray:
    hi, lo = stored(snap, head, t_hi, t_lo, 5, np.int32)
    t = np.zeros(n, np.int8)
    t[hi] = 2
    t[lo] = 1
    return t


def load_into(op, snap: dict):
    """Make oracle pool `op` hold the state of snapshot `snap` (the same
    configuration): every later oracle step then starts from the GPU's state."""
    for key in ("pages", "free_list", "table", "head_counts", "req_state", "pointers"):
        getattr(op, key)[...] = snap[key]

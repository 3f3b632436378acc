"""Decoder of the unified page format (the format stated in include/dkv.h),
written for the tests only: it reads page bytes back into per-token records
so that tests can state expectations at the level of tokens and codes.
"""
from __future__ import annotations

import numpy as np

D = 128
HI, LO = 2, 1
BITS = {HI: (8, 4), LO: (4, 2)}


def segment_offsets(t: int, kbits: int, vbits: int):
    g = 8 // vbits
    sizes = [t * D * kbits // 8, (t // g) * 128, 4 * t, 4 * t, 4 * t, 4 * t]
    offs, o = [], 0
    for s in sizes:
        offs.append(o)
        o = (o + s + 15) // 16 * 16
    return offs, offs[5] + sizes[5]


def vbit(vbits: int, f: int, e: int) -> int:
    i = f % 4
    if vbits == 4:
        return 16 * e + 4 * i
    return 16 * (e & 1) + 4 * i + 2 * (e >> 1)


def read_token(page: np.ndarray, tier: int, t: int, slot: int) -> dict:
    kb, vb = BITS[tier]
    offs, _ = segment_offsets(t, kb, vb)
    rowb = D * kb // 8
    krow = page[offs[0] + slot * rowb: offs[0] + (slot + 1) * rowb]
    if kb == 8:
        kc = krow.astype(np.int32)
    else:
        kc = np.empty(D, np.int32)
        kc[0::2] = krow & 15
        kc[1::2] = krow >> 4
    g = 8 // vb
    vrow = page[offs[1] + (slot // g) * 128: offs[1] + (slot // g + 1) * 128].view("<u4")
    e = slot % g
    vc = np.array([(int(vrow[f // 4]) >> vbit(vb, f, e)) & ((1 << vb) - 1) for f in range(D)], np.int32)
    km = page[offs[2] + 4 * slot: offs[2] + 4 * slot + 4].view("<u2")
    vm = page[offs[3] + 4 * slot: offs[3] + 4 * slot + 4].view("<u2")
    score = page[offs[4] + 4 * slot: offs[4] + 4 * slot + 4].view("<f4")[0]
    pos = page[offs[5] + 4 * slot: offs[5] + 4 * slot + 4].view("<i4")[0]
    return dict(kc=kc, vc=vc, ks=int(km[0]), kz=int(km[1]), vs=int(vm[0]), vz=int(vm[1]),
                score=float(score), pos=int(pos))


def head_tokens(snap: dict, layer: int, slot: int, kvh: int, t_hi: int, t_lo: int) -> dict:
    """All stored tokens of one head: {'hi': [records by slot], 'lo': [...]}."""
    tab = snap["table"][layer, slot, kvh]
    cnt = snap["head_counts"][layer, slot, kvh]
    L = tab.shape[0]
    out = {"hi": [], "lo": []}
    for s in range(int(cnt[0])):
        out["hi"].append(read_token(snap["pages"][tab[s // t_hi]], HI, t_hi, s % t_hi))
    for s in range(int(cnt[1])):
        out["lo"].append(read_token(snap["pages"][tab[L - 1 - s // t_lo]], LO, t_lo, s % t_lo))
    return out


def dequant(rec: dict) -> tuple[np.ndarray, np.ndarray]:
    """fp64 dequantised (k, v) of a record: scale * code + zero (exact)."""
    f = lambda b: float(np.array([b], np.uint16).view(np.float16)[0])
    k = f(rec["ks"]) * rec["kc"].astype(np.float64) + f(rec["kz"])
    v = f(rec["vs"]) * rec["vc"].astype(np.float64) + f(rec["vz"])
    return k, v


def check_invariants(snap: dict, t_hi: int, t_lo: int, n_pages: int, reclaim: bool = True):
    """Memory-management invariants: the free list's live region plus every
    table entry is a permutation of the pool (no page double-owned, none
    lost); hi and lo regions of a row never cross; page counts match token
    counts; stored positions of a head are distinct."""
    start, end = (int(x) for x in snap["pointers"])
    assert 0 <= end - start <= n_pages, (start, end)
    free_ids = [int(snap["free_list"][c % n_pages]) for c in range(start, end)]
    tab = snap["table"]
    owned = tab[tab >= 0].tolist()
    allp = sorted(free_ids + owned)
    assert allp == list(range(n_pages)), "free list + table is not a permutation of the pool"
    L = tab.shape[-1]
    cnts = snap["head_counts"]
    for idx in np.ndindex(*tab.shape[:-1]):
        row, c = tab[idx], cnts[idx]
        nhi, nlo, php, plp = (int(x) for x in c)
        assert php + plp <= L
        assert (row[:php] >= 0).all() and (row[L - plp:] >= 0).all() if plp else (row[:php] >= 0).all()
        assert (row[php:L - plp] == -1).all(), "hi and lo regions cross or leak"
        need_h, need_l = -(-nhi // t_hi), -(-nlo // t_lo)
        if reclaim:
            assert php == need_h and plp == need_l, (idx, c)
        else:
            assert php >= need_h and plp >= need_l, (idx, c)


def segment_values(snap: dict, head: tuple, t_hi: int, t_lo: int, seg: int, dtype) -> tuple[np.ndarray, np.ndarray]:
    """(hi, lo) arrays of segment `seg` (4 = score, 5 = position) of one
    head's stored slots, in slot order (head = (layer, slot, kvh))."""
    cnt = snap["head_counts"][head]
    row = snap["table"][head]
    L = row.shape[0]
    out = []
    for tier, n, t in ((HI, int(cnt[0]), t_hi), (LO, int(cnt[1]), t_lo)):
        kb, vb = BITS[tier]
        offs, _ = segment_offsets(t, kb, vb)
        vals = []
        for x in range(-(-n // t)):
            page = row[x] if tier == HI else row[L - 1 - x]
            nv = min(t, n - x * t)
            vals.append(snap["pages"][page, offs[seg]: offs[seg] + 4 * nv].view(dtype))
        out.append(np.concatenate(vals) if vals else np.zeros(0, dtype))
    return out[0], out[1]

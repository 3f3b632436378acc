"""Decoder of the unified page format (the format stated in include/dkv.h),
written for the tests only: it reads page bytes back into per-token records
so that tests can state expectations at the level of tokens and codes.
"""
from __future__ import annotations

import numpy as np

D = 128
HI, LO, MID = 2, 1, 3
# hi K8V4, lo K4V2, and the optional third level mid K8V2
BITS = {HI: (8, 4), LO: (4, 2), MID: (8, 2)}


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


def head_tokens(snap: dict, layer: int, slot: int, kvh: int, t_hi: int, t_lo: int,
                table_len: int | None = None, t_mid: int = 0) -> dict:
    """All stored tokens of one head: {'hi': [records by slot], 'lo': [...]}
    (and 'mid' when the counters have the mid level's entries; table_len is
    then the length of the two-way part of the row)."""
    tab = snap["table"][layer, slot, kvh]
    cnt = snap["head_counts"][layer, slot, kvh]
    L = tab.shape[0] if table_len is None else table_len
    out = {"hi": [], "lo": []}
    for s in range(int(cnt[0])):
        out["hi"].append(read_token(snap["pages"][tab[s // t_hi]], HI, t_hi, s % t_hi))
    for s in range(int(cnt[1])):
        out["lo"].append(read_token(snap["pages"][tab[L - 1 - s // t_lo]], LO, t_lo, s % t_lo))
    if cnt.shape[0] > 4:
        out["mid"] = [read_token(snap["pages"][tab[L + s // t_mid]], MID, t_mid, s % t_mid) for s in range(int(cnt[4]))]
    return out


def tier_page(row: np.ndarray, tier: int, k: int, table_len: int) -> int:
    """Page ID of a head's k-th page of a tier: hi from the left of the two-way
    part of the row, lo from its right, mid in the one-way part after it."""
    if tier == HI:
        return int(row[k])
    if tier == LO:
        return int(row[table_len - 1 - k])
    return int(row[table_len + k])


def dequant(rec: dict) -> tuple[np.ndarray, np.ndarray]:
    """fp64 dequantised (k, v) of a record: scale * code + zero (exact)."""
    f = lambda b: float(np.array([b], np.uint16).view(np.float16)[0])
    k = f(rec["ks"]) * rec["kc"].astype(np.float64) + f(rec["kz"])
    v = f(rec["vs"]) * rec["vc"].astype(np.float64) + f(rec["vz"])
    return k, v


def check_invariants(snap: dict, t_hi: int, t_lo: int, n_pages: int, reclaim: bool = True,
                     table_len: int | None = None, t_mid: int = 0):
    """Memory-management invariants: the free list's live region plus every
    table entry is a permutation of the pool (no page double-owned, none
    lost); hi and lo regions of a row never cross; page counts match token
    counts; stored positions of a head are distinct. With the mid level
    (counters of 8 ints) the row's one-way part after the first table_len
    entries holds exactly the mid pages, from its left."""
    start, end = (int(x) for x in snap["pointers"])
    assert 0 <= end - start <= n_pages, (start, end)
    free_ids = [int(snap["free_list"][c % n_pages]) for c in range(start, end)]
    tab = snap["table"]
    owned = tab[tab >= 0].tolist()
    allp = sorted(free_ids + owned)
    assert allp == list(range(n_pages)), "free list + table is not a permutation of the pool"
    L = tab.shape[-1] if table_len is None else table_len
    cnts = snap["head_counts"]
    mid = cnts.shape[-1] > 4
    for idx in np.ndindex(*tab.shape[:-1]):
        row, c = tab[idx], cnts[idx]
        nhi, nlo, php, plp = (int(x) for x in c[:4])
        assert php + plp <= L
        assert (row[:php] >= 0).all() and (row[L - plp:L] >= 0).all() if plp else (row[:php] >= 0).all()
        assert (row[php:L - plp] == -1).all(), "hi and lo regions cross or leak"
        need_h, need_l = -(-nhi // t_hi), -(-nlo // t_lo)
        if mid:
            nmid, pmp = int(c[4]), int(c[5])
            assert (c[6:] == 0).all()
            assert (row[L:L + pmp] >= 0).all() and (row[L + pmp:] == -1).all(), "mid region leaks"
            need_m = -(-nmid // t_mid)
            assert pmp == need_m if reclaim else pmp >= need_m, (idx, c)
        else:
            assert row.shape[0] == L
        if reclaim:
            assert php == need_h and plp == need_l, (idx, c)
        else:
            assert php >= need_h and plp >= need_l, (idx, c)


def tier_values(snap: dict, head: tuple, geo: dict, seg: int, dtype) -> dict:
    """{tier: array of segment `seg` (4 = score, 5 = position) over the tier's
    stored slots, in slot order} for one head (head = (layer, slot, kvh));
    geo: t_hi, t_lo, t_mid, table_len. Covers mid when the counters have it."""
    cnt = snap["head_counts"][head]
    row = snap["table"][head]
    L = geo["table_len"]
    tiers = [(HI, int(cnt[0]), geo["t_hi"]), (LO, int(cnt[1]), geo["t_lo"])]
    if cnt.shape[0] > 4:
        tiers.append((MID, int(cnt[4]), geo["t_mid"]))
    out = {}
    for tier, n, t in tiers:
        kb, vb = BITS[tier]
        offs, _ = segment_offsets(t, kb, vb)
        vals = []
        for x in range(-(-n // t)):
            page = tier_page(row, tier, x, L)
            nv = min(t, n - x * t)
            vals.append(snap["pages"][page, offs[seg]: offs[seg] + 4 * nv].view(dtype))
        out[tier] = np.concatenate(vals) if vals else np.zeros(0, dtype)
    return out


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

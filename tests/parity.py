"""Element-by-element comparison of two pool states (GPU export vs oracle).

Integer and page state must be identical: free-list pointers, the live part
of the free list, every table row, head counters, request state, and every
valid byte (bit, for shared value words) of every page in use. Bytes of
unused slots and segment padding are unspecified and masked out.
"""
from __future__ import annotations

import functools

import numpy as np

from tests import pagefmt


@functools.lru_cache(maxsize=None)
def valid_mask(page_bytes: int, tier: int, t: int, nvalid: int, scores: bool = True) -> np.ndarray:
    """Bit mask (uint8 per page byte) of the bits holding the first `nvalid`
    slots' data in a page of `tier` with `t` slots (score words optional)."""
    kb, vb = pagefmt.BITS[tier]
    offs, _ = pagefmt.segment_offsets(t, kb, vb)
    m = np.zeros(page_bytes, np.uint8)
    rowb = 128 * kb // 8
    m[offs[0]: offs[0] + nvalid * rowb] = 0xFF
    g = 8 // vb
    words = m[offs[1]: offs[1] + (t // g) * 128].view("<u4")
    lm = (1 << vb) - 1
    for s in range(nvalid):
        u, e = divmod(s, g)
        for f in range(128):
            words[u * 32 + f // 4] |= np.uint32(lm << pagefmt.vbit(vb, f, e))
    for seg in ((2, 3, 4, 5) if scores else (2, 3, 5)):
        m[offs[seg]: offs[seg] + 4 * nvalid] = 0xFF
    return m


def compare_states(g: dict, o: dict, t_hi: int, t_lo: int, n_pages: int, page_bytes: int,
                   heads: list | None = None, check_list: bool = True, scores: bool = True,
                   table_len: int | None = None, t_mid: int = 0):
    """Assert that GPU snapshot g equals oracle snapshot o. If `heads` is
    given, only those (layer, slot, kvh) rows and their pages are compared
    (the pool-wide list then is not). scores=False leaves the score words out
    (when the two sides computed them in different precisions). With the mid
    level, table_len is the length of the rows' two-way part and t_mid the
    mid level's tokens per page."""
    if heads is None:
        assert (g["pointers"] == o["pointers"]).all(), (g["pointers"], o["pointers"])
        if check_list:
            s, e = (int(x) for x in o["pointers"])
            idx = np.arange(s, e) % n_pages
            assert (g["free_list"][idx] == o["free_list"][idx]).all(), "free list differs"
        assert (g["table"] == o["table"]).all(), "page table differs"
        assert (g["head_counts"] == o["head_counts"]).all(), "head counters differ"
        assert (g["req_state"] == o["req_state"]).all(), "request state differs"
        heads = list(np.ndindex(*o["table"].shape[:-1]))
    L = o["table"].shape[-1] if table_len is None else table_len
    groups: dict[tuple, list] = {}
    for h in heads:
        cnt = o["head_counts"][h]
        row = o["table"][h]
        assert (g["table"][h] == row).all(), ("table row", h)
        assert (g["head_counts"][h] == cnt).all(), ("counts", h)
        tiers = [(pagefmt.HI, int(cnt[0]), t_hi), (pagefmt.LO, int(cnt[1]), t_lo)]
        if cnt.shape[0] > 4:
            tiers.append((pagefmt.MID, int(cnt[4]), t_mid))
        for tier, n, t in tiers:
            npg = -(-n // t)
            for x in range(npg):
                page = pagefmt.tier_page(row, tier, x, L)
                nvalid = min(t, n - x * t)
                groups.setdefault((tier, t, nvalid), []).append(int(page))
    for (tier, t, nvalid), pages in groups.items():
        m = valid_mask(page_bytes, tier, t, nvalid, scores)
        pg = np.asarray(pages)
        a = g["pages"][pg] & m
        b = o["pages"][pg] & m
        if not (a == b).all():
            bad = np.nonzero((a != b).any(1))[0][0]
            col = np.nonzero(a[bad] != b[bad])[0]
            raise AssertionError(f"page {pg[bad]} (tier {tier}, {nvalid} valid) differs at bytes {col[:16]}: "
                                 f"gpu {a[bad][col[:8]]} oracle {b[bad][col[:8]]}")


def within(gpu: np.ndarray, ref: np.ndarray, atol: float, rtol: float) -> tuple[bool, float]:
    """Element-wise |gpu - ref| <= atol + rtol |ref|; (holds, worst excess)."""
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    if gpu.size == 0:
        return True, -np.inf
    err = np.abs(gpu - ref) - (atol + rtol * np.abs(ref))
    return bool((err <= 0).all()), float(err.max())

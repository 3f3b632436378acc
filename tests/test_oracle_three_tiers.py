"""Pins of the oracle's third precision level (DiffKV, Compaction policy:
extensibility, more than two precision levels; Memory management, generation
workflow: further levels by combining one-way or two-way page tables).

The levels are hi K8V4, mid K8V2 and lo K4V2 (K8V2 is one of the skewed
configurations of the page's quantisation study; it keeps the keys at eight
bits, which that study found to matter more than the values). A token is hi
if I > alpha_h/N, mid if not hi and I >= alpha_m/N, lo if not mid and
I >= alpha_l/N, else pruned. Each head's table row is the two-way table (hi
pages from its left, lo pages from its right) followed by a one-way table of
mid pages.

The checks here are written from those rules alone, with nothing taken from
the oracle's code: a brute-force classification and packing of the prompt, a
hand-worked prompt with its page IDs, a step-by-step simulator of the
generation phase with the mid level (t_c and victims reach every branch), an
fp64 dense softmax over the dequantised tokens for the attention order, the
completion order of a request's pages, and planted mistakes that the
simulator must reject.
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import workloads
from tests import pagefmt
from tests.test_oracle_decode_sim import exact_score, np_dequant, np_quantize, observation_count, swap_remove

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
F32 = np.float32
HI, LO, MID = pagefmt.HI, pagefmt.LO, pagefmt.MID
NAME = {HI: "hi", MID: "mid", LO: "lo"}
RANK = {"prune": 0, "lo": 1, "mid": 2, "hi": 3}
BITS = {"hi": (8, 4), "mid": (8, 2), "lo": (4, 2)}
TIER_OF = {"hi": HI, "mid": MID, "lo": LO}


def cfg3(**kw):
    c = dict(n_layers=1, n_kv_heads=2, group_size=2, head_dim=128, page_bytes=4096, n_pages=900,
             max_requests=4, max_seq_len=400, tokens_per_hi_page=4, tokens_per_lo_page=8,
             tokens_per_mid_page=4, lo_enabled=1, mid_enabled=1, alpha_h=2.0, alpha_m=1.0, alpha_l=0.25,
             recent_window=4, obs_window=32, prompt_grant_slack=2, reclaim_in_decode=1)
    c.update(kw)
    return c


def geo(pool) -> dict:
    return dict(t_hi=pool.t_hi, t_lo=pool.t_lo, t_mid=pool.t_mid, table_len=pool.table_len)


def cls3(i, th):
    th_h, th_m, th_l = th
    if i > th_h:
        return "hi"
    if i >= th_m:
        return "mid"
    if i >= th_l:
        return "lo"
    return "prune"


def thresholds(alphas, n):
    return tuple(F32(a) / F32(n) for a in alphas)


# ------------------------------------------------------------------ prompt
def test_geometry_of_the_mid_level():
    """K8V2 page: 128-byte key rows, value rows of 4 tokens (176 bytes a
    token with its metadata, score and position); T is a multiple of 4, so a
    4096-byte page holds 20 tokens (3520 bytes; 24 would take 4224), as does a
    3584-byte page; the row composes L_e two-way entries with
    ceil(max_seq / T_mid) + 1 one-way entries; counters are 8 ints."""
    pool = oracle.Pool(cfg3(tokens_per_hi_page=0, tokens_per_lo_page=0, tokens_per_mid_page=0))
    offs, used = pagefmt.segment_offsets(20, 8, 2)
    assert pool.t_mid == 20 and list(pool.mid_off) == offs and pool.mid_used == used == 3520
    assert pagefmt.segment_offsets(24, 8, 2)[1] == 4224
    assert pool.mid_len == -(-400 // 20) + 1 and pool.row_len == pool.table_len + pool.mid_len
    assert pool.cstride == 8 and pool.head_counts.shape[-1] == 8
    p35 = oracle.Pool(cfg3(page_bytes=3584, tokens_per_hi_page=0, tokens_per_lo_page=0, tokens_per_mid_page=0))
    assert p35.t_mid == 20 and p35.t_hi == 16 and p35.t_lo == 32
    two = oracle.Pool(cfg3(mid_enabled=0))
    assert two.mid_len == 0 and two.cstride == 4 and two.row_len == two.table_len


def brute_prompt(pool, cfg, alphas, slots, lens, k, v, scores):
    """Expected per-head state after a prompt, from the rules alone: tiers by
    brute force, slots in ascending position, codes per level, pages of the
    all-hi grant taken at the list start head by head (hi from the grant's
    left, mid right after them, lo from its right), the unused middle pages
    appended at the list end."""
    H, th_ = cfg["n_kv_heads"], pool.t_hi
    W = cfg["recent_window"]
    tok0 = np.concatenate([[0], np.cumsum(lens)])
    free = list(range(cfg["n_pages"]))
    start, end = 0, cfg["n_pages"]
    grants, gl = [], 0
    for i, n0 in enumerate(lens):
        for h in range(H):
            g = -(-n0 // th_) + cfg["prompt_grant_slack"]
            grants.append(free[start + gl: start + gl + g])
            gl += g
    exp, reclaimed = {}, []
    for i, (s, n0) in enumerate(zip(slots, lens)):
        for h in range(H):
            th = thresholds(alphas[h], n0)
            tiers = {"hi": [], "mid": [], "lo": []}
            for j in range(n0):
                S = F32(scores[tok0[i] + j, h])
                c = max(1, min(32, n0 - j))
                t = "hi" if j >= n0 - W else cls3(F32(S / F32(c)), th)
                if t != "prune":
                    tiers[t].append(j)
            grant = grants[i * H + h]
            php = -(-len(tiers["hi"]) // pool.t_hi)
            pmp = -(-len(tiers["mid"]) // pool.t_mid)
            plp = -(-len(tiers["lo"]) // pool.t_lo)
            pages = {"hi": grant[:php], "mid": grant[php:php + pmp], "lo": grant[len(grant) - plp:][::-1]}
            reclaimed += grant[php + pmp:len(grant) - plp]
            exp[(0, s, h)] = (tiers, pages)
    return exp, start + gl, end + len(reclaimed), reclaimed


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prompt_three_levels_brute_force(seed):
    cfg = cfg3()
    H = cfg["n_kv_heads"]
    slots, lens = [0, 2, 3], [37, 120, 9]
    n_tok = sum(lens)
    pool = oracle.Pool(cfg)
    alphas = [(2.0, 1.0, 0.25), (1.5, 0.7, 0.4)]
    assert pool.set_thresholds(0, [a[0] for a in alphas], [a[2] for a in alphas]) == 0
    assert pool.set_mid_thresholds(0, [a[1] for a in alphas]) == 0
    k = workloads.random_fp16((n_tok, H, 128), 10 + seed)
    v = workloads.random_fp16((n_tok, H, 128), 20 + seed)
    scores = workloads.given_scores(n_tok, H, seed=30 + seed).astype(F32)
    # a few importances exactly on each threshold (both sides of every closure)
    rng = np.random.default_rng(seed)
    tok0 = np.concatenate([[0], np.cumsum(lens)])
    for i, n0 in enumerate(lens):
        for h in range(H):
            th = thresholds(alphas[h], n0)
            for j in rng.choice(max(1, n0 - cfg["recent_window"]), size=min(6, n0), replace=True):
                x = exact_score(th[int(rng.integers(0, 3))], max(1, min(32, n0 - int(j))))
                if x is not None:
                    scores[tok0[i] + j, h] = x
    assert pool.prompt(0, slots, lens, k, v, scores_in=scores) == 0
    snap = pool.snapshot()
    exp, start, end, reclaimed = brute_prompt(pool, cfg, alphas, slots, lens, k, v, scores)
    assert tuple(int(x) for x in snap["pointers"]) == (start, end)
    assert [int(snap["free_list"][(cfg["n_pages"] + x) % cfg["n_pages"]]) for x in range(len(reclaimed))] == reclaimed
    seen_tiers = set()
    for (layer, s, h), (tiers, pages) in exp.items():
        cnt = snap["head_counts"][layer, s, h]
        assert tuple(int(x) for x in cnt) == (len(tiers["hi"]), len(tiers["lo"]), len(pages["hi"]),
                                              len(pages["lo"]), len(tiers["mid"]), len(pages["mid"]), 0, 0)
        row = snap["table"][layer, s, h]
        for name, tier in TIER_OF.items():
            assert [pagefmt.tier_page(row, tier, x, pool.table_len) for x in range(len(pages[name]))] == pages[name]
        i = slots.index(s)
        recs = pagefmt.head_tokens(snap, layer, s, h, pool.t_hi, pool.t_lo, pool.table_len, pool.t_mid)
        for name in ("hi", "mid", "lo"):
            assert [r["pos"] for r in recs[name]] == tiers[name], (s, h, name)
            kb, vb = BITS[name]
            for r in recs[name]:
                t = tok0[i] + r["pos"]
                kc, ks, kz = np_quantize(k[t, h].astype(F32), kb)
                vc, vs, vz = np_quantize(v[t, h].astype(F32), vb)
                assert (r["kc"] == kc).all() and (r["vc"] == vc).all() and (r["ks"], r["kz"], r["vs"], r["vz"]) == (
                    ks, kz, vs, vz), (s, h, name, r["pos"])
                assert np.float32(r["score"]) == scores[t, h]
            if tiers[name]:
                seen_tiers.add(name)
    assert seen_tiers == {"hi", "mid", "lo"}
    pagefmt.check_invariants(snap, pool.t_hi, pool.t_lo, cfg["n_pages"], table_len=pool.table_len, t_mid=pool.t_mid)


def test_prompt_worked_example():
    """One head of 14 tokens, W = 2, T_hi = 2, T_mid = T_lo = 4, slack 2:
    grant ceil(14/2) + 2 = 9 pages, 0..8. Importances (c = 14 - j for every j
    here, all observation queries): positions 0, 5 hi (above 2/14); 1, 2, 6
    mid (in [1/14, 2/14]); 3, 7, 8, 9, 10 lo (in [0.25/14, 1/14)); 4, 11
    pruned; 12, 13 the window (hi). hi: 0, 5, 12, 13 -> pages 0, 1; mid: 1,
    2, 6 -> page 2; lo: 3, 7, 8, 9, 10 -> pages 8, 7 (from the right); pages
    3, 4, 5, 6 go back to the list end in that order."""
    cfg = cfg3(n_kv_heads=1, group_size=1, n_pages=32, recent_window=2, tokens_per_hi_page=2,
               tokens_per_mid_page=4, tokens_per_lo_page=4)
    pool = oracle.Pool(cfg)
    imp = {0: 3.0, 5: 2.5, 1: 1.0, 2: 1.5, 6: 2.0, 3: 0.25, 7: 0.5, 8: 0.9, 9: 0.3, 10: 0.99, 4: 0.2, 11: 0.0,
           12: 0.0, 13: 0.0}
    want_cls = {0: "hi", 5: "hi", 1: "mid", 2: "mid", 6: "mid", 3: "lo", 7: "lo", 8: "lo", 9: "lo", 10: "lo",
                4: "prune", 11: "prune"}
    scores = np.zeros((14, 1), F32)
    for j, a in imp.items():
        s = exact_score(F32(a) / F32(14), 14 - j) if a > 0 else F32(0.0)
        if s is None:           # no fp32 score gives that importance exactly: the nearest one
            s = F32(F32(a) / F32(14) * F32(14 - j))
        scores[j, 0] = s
        if j in want_cls:       # the example's classes hold for the scores written
            assert cls3(F32(s / F32(14 - j)), thresholds((2.0, 1.0, 0.25), 14)) == want_cls[j], j
    k = workloads.random_fp16((14, 1, 128), 1)
    v = workloads.random_fp16((14, 1, 128), 2)
    assert pool.prompt(0, [0], [14], k, v, scores_in=scores) == 0
    row = pool.table[0, 0, 0]
    L = pool.table_len
    assert L == 200 + 1 and pool.mid_len == 100 + 1
    assert list(row[:2]) == [0, 1] and list(row[L:L + 1]) == [2] and list(row[L - 2:L]) == [7, 8]
    assert (row[2:L - 2] == -1).all() and (row[L + 1:] == -1).all()
    assert list(pool.head_counts[0, 0, 0]) == [4, 5, 2, 2, 3, 1, 0, 0]
    assert list(pool.pointers) == [9, 36] and list(pool.free_list[[0, 1, 2, 3]]) == [3, 4, 5, 6]
    recs = pagefmt.head_tokens(pool.snapshot(), 0, 0, 0, 2, 4, L, 4)
    assert [r["pos"] for r in recs["hi"]] == [0, 5, 12, 13]
    assert [r["pos"] for r in recs["mid"]] == [1, 2, 6]
    assert [r["pos"] for r in recs["lo"]] == [3, 7, 8, 9, 10]


def test_prompt_table_full_with_one_slack_page():
    """Three partial pages can exceed the all-hi grant of ceil(N0/T_hi) + 1:
    N0 = 4, T_hi = T_mid = T_lo = 4, W = 1, importances (thresholds 2/4, 1/4,
    0.25/4) put positions 2, 3 hi, 0 mid and 1 lo: 3 pages against a grant of
    2. With two slack pages the prompt fits."""
    cfg = cfg3(n_kv_heads=1, group_size=1, n_pages=32, recent_window=1, tokens_per_hi_page=4,
               tokens_per_mid_page=4, tokens_per_lo_page=4, prompt_grant_slack=1)
    pool = oracle.Pool(cfg)
    scores = np.array([[1.2], [0.3], [2.0], [0.0]], F32)    # I = 0.3, 0.1, 1.0 (c = 4, 3, 2)
    k = workloads.random_fp16((4, 1, 128), 1)
    assert pool.prompt(0, [0], [4], k, k, scores_in=scores) == oracle.ERR["TABLE_FULL"]
    assert list(pool.pointers) == [0, 32] and (pool.table == -1).all()
    pool2 = oracle.Pool(dict(cfg, prompt_grant_slack=2))
    assert pool2.prompt(0, [0], [4], k, k, scores_in=scores) == 0
    assert list(pool2.head_counts[0, 0, 0][:6]) == [2, 1, 1, 1, 1, 1]


# -------------------------------------------------------------- generation
class Head3:
    def __init__(self, tiers, pages):
        self.t = tiers                  # name -> positions in slot order
        self.np = pages                 # name -> page count
        self.seen, self.score = {}, {}


def sim_step3(h: Head3, n: int, W: int, th):
    """One generation step of one head with three levels, literally: the new
    token enters hi; t_c (position n - W - 1) is classified; if it stays hi,
    the least important hi token outside the window is the victim; if it
    moves to mid or lo, the least important token of that level (t_c
    included) is; if pruned, nothing more. A victim that classifies at its
    own level or above stays; one that classifies lower moves to the end of
    that level (re-quantised) or is pruned. Removal moves the level's last
    slot into the hole. Returns {position: level it was re-quantised from}."""
    imp = lambda p: F32(h.score[p]) / F32(max(1, h.seen[p]))
    key = lambda p: (imp(p), p)
    h.t["hi"].append(n - 1)
    h.score[n - 1], h.seen[n - 1] = F32(0.0), 0
    moved = {}
    pc = n - W - 1
    branch = None
    if pc >= 0:
        c = cls3(imp(pc), th)
        vt = None
        if c == "prune":
            swap_remove(h.t["hi"], h.t["hi"].index(pc))
        elif c == "hi":
            vt = "hi"
        else:
            swap_remove(h.t["hi"], h.t["hi"].index(pc))
            h.t[c].append(pc)
            moved[pc] = "hi"
            vt = c
        branch = (c, None)
        if vt is not None:
            lst = h.t[vt]
            cand = [x for x in range(len(lst)) if vt != "hi" or lst[x] < n - W]
            xv = min(cand, key=lambda x: key(lst[x]))
            pv = lst[xv]
            cv = cls3(imp(pv), th)
            branch = (c, cv if RANK[cv] < RANK[vt] else "keep")
            if RANK[cv] < RANK[vt]:
                swap_remove(lst, xv)
                if cv != "prune":
                    h.t[cv].append(pv)
                    moved[pv] = moved.get(pv, vt)
    live = set(h.t["hi"]) | set(h.t["mid"]) | set(h.t["lo"])
    for p in list(h.score):
        if p not in live:
            del h.score[p]
            h.seen.pop(p, None)
    return moved, branch


LEVELS = ["zero", "below_l", "at_l", "l_m", "at_m", "m_h", "at_h", "above_h", "high"]


def design3(h: Head3, n: int, W: int, th, rng):
    """Scores for the coming step reaching one branch (at random), with
    importances on and next to every threshold and ties at the minimum."""
    th_h, th_m, th_l = th
    val = {"zero": F32(0.0), "below_l": F32(th_l * F32(0.5)), "at_l": th_l, "l_m": F32((th_l + th_m) * F32(0.5)),
           "at_m": th_m, "m_h": F32((th_m + th_h) * F32(0.5)), "at_h": th_h, "above_h": F32(th_h * F32(1.25)),
           "high": F32(th_h * F32(4))}
    seen = lambda p: max(1, h.seen[p])

    def put(p, lvl):
        s = exact_score(val[lvl], seen(p))
        h.score[p] = s if s is not None else F32(val[lvl] * F32(seen(p)))

    def above(lvl):
        i = LEVELS.index(lvl)
        return LEVELS[rng.integers(i + 1, len(LEVELS))] if i + 1 < len(LEVELS) else lvl

    for p in h.t["hi"] + h.t["mid"] + h.t["lo"]:
        put(p, LEVELS[rng.integers(0, len(LEVELS))])
    window = [p for p in h.t["hi"] if p >= n - W]
    for p in window:
        h.score[p] = F32(0.0)
    pc = n - W - 1
    if pc < 0:
        return
    branch = ["hi", "mid", "lo", "prune"][rng.choice(4, p=[0.4, 0.3, 0.2, 0.1])]
    if branch == "prune":
        put(pc, ["zero", "below_l"][rng.integers(0, 2)])
        return
    if branch == "hi":
        put(pc, ["above_h", "high"][rng.integers(0, 2)])
        lst = [p for p in h.t["hi"] if p < n - W and p != pc]
        floor = LEVELS[rng.integers(0, 8)]
    elif branch == "mid":
        put(pc, ["at_m", "m_h", "at_h"][rng.integers(0, 3)])
        lst = list(h.t["mid"])
        floor = LEVELS[rng.integers(0, 6)]
    else:
        put(pc, ["at_l", "l_m"][rng.integers(0, 2)])
        lst = list(h.t["lo"])
        floor = LEVELS[rng.integers(0, 4)]
    for p in lst:
        put(p, above(floor))
    kk = min(len(lst), int(rng.integers(1, 4)))
    for p in (rng.choice(lst, size=kk, replace=False) if kk else []):
        put(int(p), floor)


def write_score3(pool, head, h: Head3, pos: int, value):
    layer, slot, kvh = head
    row = pool.table[layer, slot, kvh]
    for name, tier, t, off in (("hi", HI, pool.t_hi, pool.hi_off), ("mid", MID, pool.t_mid, pool.mid_off),
                               ("lo", LO, pool.t_lo, pool.lo_off)):
        if pos in h.t[name]:
            s = h.t[name].index(pos)
            page = pagefmt.tier_page(row, tier, s // t, pool.table_len)
            o = off[4] + 4 * (s % t)
            pool.pages[page, o:o + 4] = np.array([value], F32).view(np.uint8)
            return
    raise AssertionError(pos)


def record(snap, head, pool, name, slot):
    t = {"hi": pool.t_hi, "mid": pool.t_mid, "lo": pool.t_lo}[name]
    page = pagefmt.tier_page(snap["table"][head], TIER_OF[name], slot // t, pool.table_len)
    return pagefmt.read_token(snap["pages"][page], TIER_OF[name], t, slot % t)


def same(a, b):
    return all((np.asarray(a[x]) == np.asarray(b[x])).all() for x in ("kc", "vc", "ks", "kz", "vs", "vz", "pos")) \
        and np.float32(a["score"]).view(np.uint32) == np.float32(b["score"]).view(np.uint32)


def run_generation(cfg, alphas, steps, seed, check_codes=True):
    H, W = cfg["n_kv_heads"], cfg["recent_window"]
    slots, lens = [0, 1, 3], [40, 3, 70]
    n_tok = sum(lens)
    pool = oracle.Pool(cfg)
    assert pool.set_thresholds(0, [a[0] for a in alphas], [a[2] for a in alphas]) == 0
    assert pool.set_mid_thresholds(0, [a[1] for a in alphas]) == 0
    k = workloads.random_fp16((n_tok, H, 128), 5)
    vv = workloads.random_fp16((n_tok, H, 128), 6)
    assert pool.prompt(0, slots, lens, k, vv, scores_in=workloads.given_scores(n_tok, H, seed=7)) == 0
    rng = np.random.default_rng(seed)
    snap = pool.snapshot()
    g = geo(pool)
    sim, N = {}, {s: n0 for s, n0 in zip(slots, lens)}
    for s, n0 in zip(slots, lens):
        for kvh in range(H):
            hd = (0, s, kvh)
            pos = pagefmt.tier_values(snap, hd, g, 5, np.int32)
            cnt = snap["head_counts"][hd]
            h = Head3({n: [int(x) for x in pos[TIER_OF[n]]] for n in ("hi", "mid", "lo")},
                      {"hi": int(cnt[2]), "lo": int(cnt[3]), "mid": int(cnt[5])})
            for p in h.t["hi"] + h.t["mid"] + h.t["lo"]:
                h.seen[p] = observation_count(p, n0)
            sim[(s, kvh)] = h
    branches = set()
    for step in range(steps):
        for s in slots:
            n = N[s] + 1
            for kvh in range(H):
                h = sim[(s, kvh)]
                design3(h, n, W, thresholds(alphas[kvh], n), rng)
                for p in h.t["hi"] + h.t["mid"] + h.t["lo"]:
                    write_score3(pool, (0, s, kvh), h, p, h.score[p])
        before = pool.snapshot()
        start, end = (int(x) for x in before["pointers"])
        kn = workloads.random_fp16((len(slots), H, 128), 1000 + step)
        vn = workloads.random_fp16((len(slots), H, 128), 2000 + step)
        pred, aoff, freed = {}, 0, []
        for i, s in enumerate(slots):
            n = N[s] + 1
            for kvh in range(H):
                h = sim[(s, kvh)]
                old = {x: list(h.t[x]) for x in h.t}
                moved, branch = sim_step3(h, n, W, thresholds(alphas[kvh], n))
                branches.add(branch)
                ids = {}
                row = before["table"][(0, s, kvh)]
                for name in ("hi", "lo", "mid"):       # allocation order of a head
                    t = {"hi": pool.t_hi, "mid": pool.t_mid, "lo": pool.t_lo}[name]
                    need = -(-len(h.t[name]) // t)
                    new = max(0, need - h.np[name])
                    ids[name] = [int(before["free_list"][(start + aoff + x) % cfg["n_pages"]]) for x in range(new)]
                    aoff += new
                for name in ("hi", "lo", "mid"):
                    t = {"hi": pool.t_hi, "mid": pool.t_mid, "lo": pool.t_lo}[name]
                    need = -(-len(h.t[name]) // t)
                    for x in range(max(0, h.np[name] - need)):
                        freed.append(pagefmt.tier_page(row, TIER_OF[name], h.np[name] - 1 - x, pool.table_len))
                pred[(s, kvh)] = (old, moved, ids, i)
        assert pool.decode(0, slots, kn, vn) == 0
        after = pool.snapshot()
        assert int(after["pointers"][0]) == start + aoff
        assert int(after["pointers"][1]) == end + len(freed)
        assert [int(after["free_list"][(end + x) % cfg["n_pages"]]) for x in range(len(freed))] == freed
        for s in slots:
            N[s] += 1
        for (s, kvh), (old, moved, ids, i) in pred.items():
            h = sim[(s, kvh)]
            hd = (0, s, kvh)
            ctx = f"step {step} slot {s} kvh {kvh}"
            pos = pagefmt.tier_values(after, hd, g, 5, np.int32)
            sc = pagefmt.tier_values(after, hd, g, 4, np.float32)
            row = after["table"][hd]
            for name in ("hi", "mid", "lo"):
                assert pos[TIER_OF[name]].tolist() == h.t[name], (ctx, name, pos[TIER_OF[name]].tolist(), h.t[name])
                assert sc[TIER_OF[name]].tolist() == [float(h.score[p]) for p in h.t[name]], (ctx, name)
                t = {"hi": pool.t_hi, "mid": pool.t_mid, "lo": pool.t_lo}[name]
                need = -(-len(h.t[name]) // t)
                got_new = [pagefmt.tier_page(row, TIER_OF[name], h.np[name] + x, pool.table_len)
                           for x in range(len(ids[name]))]
                assert got_new == ids[name], (ctx, name)
                h.np[name] = need
            cnt = after["head_counts"][hd]
            assert tuple(int(x) for x in cnt) == (len(h.t["hi"]), len(h.t["lo"]), h.np["hi"], h.np["lo"],
                                                  len(h.t["mid"]), h.np["mid"], 0, 0), ctx
            if not check_codes:
                continue
            for name in ("hi", "mid", "lo"):
                kb, vb = BITS[name]
                for x, p in enumerate(h.t[name]):
                    if x < len(old[name]) and old[name][x] == p:
                        continue
                    got = record(after, hd, pool, name, x)
                    if p == N[s] - 1:
                        kc, ks, kz = np_quantize(kn[i, kvh].astype(F32), 8)
                        vc, vs, vz = np_quantize(vn[i, kvh].astype(F32), 4)
                        want = dict(kc=kc, vc=vc, ks=ks, kz=kz, vs=vs, vz=vz, score=0.0, pos=p)
                    elif p in moved:
                        src = record(before, hd, pool, moved[p], old[moved[p]].index(p))
                        kc, ks, kz = np_quantize(np_dequant(src["kc"], src["ks"], src["kz"]), kb)
                        vc, vs, vz = np_quantize(np_dequant(src["vc"], src["vs"], src["vz"]), vb)
                        want = dict(kc=kc, vc=vc, ks=ks, kz=kz, vs=vs, vz=vz, score=src["score"], pos=p)
                    else:
                        want = record(before, hd, pool, name, old[name].index(p))
                    assert same(got, want), (ctx, "slot content", name, x, p)
        pagefmt.check_invariants(after, pool.t_hi, pool.t_lo, cfg["n_pages"], table_len=pool.table_len,
                                 t_mid=pool.t_mid)
        for s in slots:
            pool.req_state[0, s, 3] += 1
            for kvh in range(H):
                for p in sim[(s, kvh)].t["hi"] + sim[(s, kvh)].t["mid"] + sim[(s, kvh)].t["lo"]:
                    sim[(s, kvh)].seen[p] += 1
    return branches


VARIANTS3 = {
    "per_head": dict(alphas=[(2.0, 1.0, 0.25), (1.2, 0.8, 0.5)], cfg=dict()),
    "w1_no_reclaim": dict(alphas=[(2.0, 1.0, 0.25), (2.0, 1.0, 0.25)], cfg=dict(recent_window=1, reclaim_in_decode=0)),
}


@pytest.mark.parametrize("variant", list(VARIANTS3))
def test_generation_three_levels_matches_simulator(variant):
    v = VARIANTS3[variant]
    branches = run_generation(cfg3(**v["cfg"]), v["alphas"], 70, zlib.crc32(variant.encode()))
    want = {("prune", None), ("hi", "keep"), ("hi", "mid"), ("hi", "lo"), ("hi", "prune"), ("mid", "keep"),
            ("mid", "lo"), ("mid", "prune"), ("lo", "keep"), ("lo", "prune")}
    assert want <= branches, want - branches


# ----------------------------------------------------------------- attention
def test_attention_over_three_levels_is_dense_softmax():
    """fp64 attention of the oracle equals a dense softmax over every stored
    token's dequantised K and V (hi, mid and lo alike), and its score update
    adds the group maximum of each token's probability, in the order hi slots,
    mid slots, lo slots."""
    cfg = cfg3(group_size=3)
    branches = None
    pool = oracle.Pool(cfg)
    H, G = 2, 3
    lens = [150, 61]
    k = workloads.random_fp16((sum(lens), H, 128), 3)
    v = workloads.random_fp16((sum(lens), H, 128), 4)
    assert pool.prompt(0, [0, 1], lens, k, v, scores_in=workloads.given_scores(sum(lens), H, seed=9)) == 0
    q = workloads.random_fp16((2, H * G, 128), 11)
    before = pool.snapshot()
    rc, out = pool.attention(0, [0, 1], q, update_scores=True)
    assert rc == 0
    after = pool.snapshot()
    for i in range(2):
        for h in range(H):
            recs = pagefmt.head_tokens(before, 0, i, h, pool.t_hi, pool.t_lo, pool.table_len, pool.t_mid)
            order = recs["hi"] + recs["mid"] + recs["lo"]
            assert recs["mid"], "no mid token"
            kd = np.stack([pagefmt.dequant(r)[0] for r in order])
            vd = np.stack([pagefmt.dequant(r)[1] for r in order])
            qd = q[i, h * G:(h + 1) * G].astype(np.float64)
            lg = qd @ kd.T / np.sqrt(128.0)
            p = np.exp(lg - lg.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            np.testing.assert_allclose(out[i, h * G:(h + 1) * G], p @ vd, rtol=1e-12, atol=1e-12)
            newrecs = pagefmt.head_tokens(after, 0, i, h, pool.t_hi, pool.t_lo, pool.table_len, pool.t_mid)
            new_scores = [r["score"] for r in newrecs["hi"] + newrecs["mid"] + newrecs["lo"]]
            want = [float(np.float32(np.float64(np.float32(r["score"])) + pm)) for r, pm in zip(order, p.max(0))]
            assert new_scores == want
    assert branches is None


def test_free_request_order_three_levels():
    """A finished request's pages go to the list end head by head: hi pages
    left to right, lo pages from the outermost in, then mid pages left to
    right; rows and counters are cleared."""
    cfg = cfg3()
    pool = oracle.Pool(cfg)
    H = 2
    lens = [90, 33]
    k = workloads.random_fp16((sum(lens), H, 128), 3)
    assert pool.prompt(0, [1, 2], lens, k, k, scores_in=workloads.given_scores(sum(lens), H, seed=2)) == 0
    before = pool.snapshot()
    end = int(before["pointers"][1])
    want = []
    for h in range(H):
        row, cnt = before["table"][0, 1, h], before["head_counts"][0, 1, h]
        want += [pagefmt.tier_page(row, HI, x, pool.table_len) for x in range(int(cnt[2]))]
        want += [pagefmt.tier_page(row, LO, x, pool.table_len) for x in range(int(cnt[3]))]
        want += [pagefmt.tier_page(row, MID, x, pool.table_len) for x in range(int(cnt[5]))]
    assert pool.free_request(1) == 0
    after = pool.snapshot()
    assert int(after["pointers"][1]) == end + len(want)
    assert [int(after["free_list"][(end + x) % cfg["n_pages"]]) for x in range(len(want))] == want
    assert (after["table"][0, 1] == -1).all() and (after["head_counts"][0, 1] == 0).all()
    pagefmt.check_invariants(after, pool.t_hi, pool.t_lo, cfg["n_pages"], table_len=pool.table_len, t_mid=pool.t_mid)


# ------------------------------------------------------------ planted mistakes
MUTANTS3 = {
    "mid_threshold_exclusive": ("imp >= am / (float)n) return TIER_MID;", "imp > am / (float)n) return TIER_MID;"),
    "mid_pages_not_reclaimed_past": ("for (int x = php + pmp; x < grant[hd] - plp; x++) {",
                                     "for (int x = php + pmp + 1; x < grant[hd] - plp; x++) {"),
    "mid_from_grant_start": ("put_token(page_ptr(p, gp[hd][php + rm / tm])", "put_token(page_ptr(p, gp[hd][rm / tm])"),
    "requant_skipped": ("else requant(&t, &p->tg[tier], &recs[tier][x]);",
                        "else { recs[tier][x] = t; recs[tier][x].kc[0] ^= 0; }"),
    "tc_not_a_victim_candidate": ("vt == TIER_HI ? n - c->window : 0x7fffffff)", "vt == TIER_HI ? n - c->window : pc)"),
    "mid_pages_freed_after_lo_reversed": (
        "for (int x = 0; x < cn[5]; x++) p->list[(p->ptr[1]++) % c->n_pages] = row[p->table_len + x];",
        "for (int x = cn[5] - 1; x >= 0; x--) p->list[(p->ptr[1]++) % c->n_pages] = row[p->table_len + x];"),
    "mid_thresholds_of_head0": ("const float am = p->alpha_mid[hx];",
                                "const float am = p->alpha_mid[(size_t)layer * H];"),
}


@pytest.mark.slow
def test_planted_mistakes_three_levels_are_caught():
    """Each planted mistake in a copy of the oracle (CPU only) fails one of the
    three-level pins; the unchanged copy passes them."""
    src = open(os.path.join(ROOT, "oracle", "dkv_oracle.c")).read()
    with tempfile.TemporaryDirectory() as tmp:
        def run(name, text):
            c_path, so_path = os.path.join(tmp, f"{name}.c"), os.path.join(tmp, f"{name}.so")
            open(c_path, "w").write(text)
            subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                            "-o", so_path, c_path, "-lm"], check=True)
            env = dict(os.environ, DKV_ORACLE_LIB=so_path)
            r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                                os.path.join(HERE, "test_oracle_three_tiers.py"), "-k",
                                "brute_force or worked_example or matches_simulator or free_request_order"],
                               cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
            return r.returncode
        for name, (old, new) in MUTANTS3.items():
            assert src.count(old) == 1, f"mutation site of {name} not found once in the oracle"
        jobs = [("unchanged", src)] + [(name, src.replace(old, new)) for name, (old, new) in MUTANTS3.items()]
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
            rcs = dict(zip([j[0] for j in jobs], ex.map(lambda j: run(*j), jobs)))
        assert rcs.pop("unchanged") == 0
        survived = [name for name, rc in rcs.items() if rc == 0]
        assert not survived, f"planted mistakes not caught: {survived}"

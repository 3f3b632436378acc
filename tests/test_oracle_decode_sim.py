"""Pin of the oracle's generation-phase step against an independent
step-by-step simulator (DiffKV, Compaction policy: generation-phase logic and
the algorithm flow; Memory management: generation-phase workflow).

The simulator here keeps, for every head, the explicit slot lists of the
positions each tier stores, and a literal count of the queries that have seen
each stored token: the prompt's observation queries at or after it, then one
per score update made while it was stored. Before every step the test writes
crafted scores and the update counter into the oracle's own state. The scores
put importances exactly on the thresholds, just off them, and tie several
tokens at the minimum, so that every branch of the flow is taken: t_c kept
high with its victim kept, demoted or pruned; t_c demoted with the low-tier
victim pruned or kept; t_c pruned. Tokens inside the recent window get the
lowest score of all, so a victim search that looked into the window would pick
one of them.

After each step the oracle must store exactly the predicted positions, slot by
slot, in both tiers, with the predicted scores; the new, moved and demoted
tokens must carry the predicted codes (a demoted token is re-quantised from
its dequantised high-precision values by a numpy codec written here from the
quantisation formula of the Background section); page counts, table rows and
the list start must follow.

test_planted_mistakes_are_caught builds copies of the oracle with one
plausible mistake each (a victim by argmax, `>=` where `>` is meant, a query
count off by one, the window ignored, ...) and requires this simulator to
reject every one of them.
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import pytest

import oracle
import workloads
from tests import pagefmt

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
F32 = np.float32


# ------------------------------------------------------------ numpy codec
def np_quantize(x: np.ndarray, bits: int):
    """Asymmetric min/max quantisation of one fp32 vector: fp16 scale
    (max - min) / (2^bits - 1) and zero min (a -0 zero taken as +0), codes
    round-half-even((x - z) / s) clamped to [0, 2^bits - 1], all in fp32."""
    x = np.asarray(x, F32)
    L = (1 << bits) - 1
    mn, mx = x.min(), x.max()
    if mn == 0:
        mn = F32(0.0)
    s16 = np.float16(F32(mx - mn) / F32(L))
    z16 = np.float16(mn)
    s, z = F32(s16), F32(z16)
    if s == 0:
        codes = np.zeros(x.size, np.int32)
    else:
        inv = F32(1.0) / s
        codes = np.clip(np.rint((x - z) * inv), 0, L).astype(np.int32)
    return codes, int(s16.view(np.uint16)), int(z16.view(np.uint16))


def np_dequant(codes, s_bits: int, z_bits: int) -> np.ndarray:
    """fp32 of s * code + z with one rounding (the fp64 product and sum are exact)."""
    s = float(np.array([s_bits], np.uint16).view(np.float16)[0])
    z = float(np.array([z_bits], np.uint16).view(np.float16)[0])
    return (s * np.asarray(codes, np.float64) + z).astype(F32)


# -------------------------------------------------------------- simulator
@dataclass
class SimHead:
    hi: list                     # positions, hi slot order
    lo: list                     # positions, lo slot order
    php: int
    plp: int
    seen: dict = field(default_factory=dict)    # position -> queries that saw it
    score: dict = field(default_factory=dict)   # position -> fp32 score


def observation_count(j: int, n0: int, obs: int = 32) -> int:
    """Observation queries (the prompt's last `obs` positions) at or after j."""
    return sum(1 for p in range(max(0, n0 - obs), n0) if p >= j)


def swap_remove(a: list, x: int):
    a[x] = a[-1]
    a.pop()


def sim_step(h: SimHead, n: int, W: int, th_h, th_l, lo_enabled: bool):
    """One generation-phase step of one head, literally: (1) the new token
    (position n - 1) enters the high tier; (2) t_c, the token leaving the
    window, is classified; if high, the least important high token outside
    the window is kept, demoted or pruned; if low, t_c moves to the low tier
    and the least important low token is pruned below alpha_l / N; if pruned,
    t_c is removed. Removal moves the tier's last slot into the hole. Returns
    the set of demoted positions."""
    imp = lambda p: F32(h.score[p]) / F32(max(1, h.seen[p]))
    key = lambda p: (imp(p), p)

    def cls(i):
        if lo_enabled:
            return "hi" if i > th_h else ("lo" if i >= th_l else "prune")
        return "hi" if i >= th_l else "prune"

    h.hi.append(n - 1)
    h.score[n - 1] = F32(0.0)
    h.seen[n - 1] = 0
    demoted = set()
    pc = n - W - 1
    if pc >= 0:
        xc = h.hi.index(pc)
        c = cls(imp(pc))
        if c == "hi":
            cand = [x for x in range(len(h.hi)) if h.hi[x] < n - W]
            xv = min(cand, key=lambda x: key(h.hi[x]))
            pv = h.hi[xv]
            iv = imp(pv)
            keep = iv > th_h if lo_enabled else iv >= th_l
            if not keep:
                swap_remove(h.hi, xv)
                if lo_enabled and iv >= th_l:
                    h.lo.append(pv)
                    demoted.add(pv)
        elif c == "lo":
            swap_remove(h.hi, xc)
            h.lo.append(pc)
            demoted.add(pc)
            xv = min(range(len(h.lo)), key=lambda x: key(h.lo[x]))
            if imp(h.lo[xv]) < th_l:
                swap_remove(h.lo, xv)
        else:
            swap_remove(h.hi, xc)
    live = set(h.hi) | set(h.lo)
    for p in list(h.score):
        if p not in live:
            del h.score[p]
            h.seen.pop(p, None)
    return demoted


# ------------------------------------------------------------ score design
def exact_score(target, c: int):
    """An fp32 score S >= 0 with fp32(S / c) == target exactly, or None."""
    target, c32 = F32(target), F32(c)
    s = F32(target * c32)
    cands = [s]
    up = dn = s
    for _ in range(8):
        up = np.nextafter(up, F32(np.inf))
        dn = np.nextafter(dn, F32(-np.inf))
        cands += [up, dn]
    for x in cands:
        if x >= 0 and F32(x / c32) == target:
            return F32(x)
    return None


def design_scores(h: SimHead, n: int, W: int, th_h, th_l, lo_enabled: bool, rng) -> dict:
    """Scores for every stored token of one head for the coming step, chosen
    to reach one branch of the flow (at random) with importances on or next
    to the thresholds and ties at the minimum."""
    levels = {"zero": F32(0.0), "below_l": F32(th_l * F32(0.5)), "at_l": th_l,
              "mid": F32((th_l + th_h) * F32(0.5)) if np.isfinite(th_h) else F32(th_l * F32(3)),
              "at_h": th_h, "above_h": F32(th_h * F32(1.25)), "high": F32(th_h * F32(4))}
    order = ["zero", "below_l", "at_l", "mid", "at_h", "above_h", "high"]
    seen = lambda p: max(1, h.seen[p])

    def put(p, lvl):
        s = exact_score(levels[lvl], seen(p)) if np.isfinite(levels[lvl]) else None
        if s is None:                     # no exact fp32 score: a value well inside the level
            s = F32(F32(levels[lvl]) * F32(seen(p))) if np.isfinite(levels[lvl]) else F32(1e30)
        h.score[p] = s

    def above(lvl):
        return order[rng.integers(order.index(lvl) + 1, len(order))] if lvl != "high" else "high"

    pc = n - W - 1
    window = [p for p in h.hi if p >= n - W]
    elig = [p for p in h.hi if p < n - W and p != pc]
    for p in h.hi + h.lo:
        put(p, order[rng.integers(0, len(order))])
    for p in window:
        h.score[p] = F32(0.0)
    if pc < 0:
        return {}
    if lo_enabled:
        branch = ["hi", "lo", "prune"][rng.choice(3, p=[0.5, 0.35, 0.15])]
    else:
        branch = ["hi", "prune"][rng.choice(2, p=[0.75, 0.25])]
    if branch == "prune":
        put(pc, ["zero", "below_l"][rng.integers(0, 2)])
        return {"branch": branch}
    if branch == "hi":
        put(pc, ["above_h", "high"][rng.integers(0, 2)] if lo_enabled
            else ["at_l", "mid", "at_h", "above_h"][rng.integers(0, 4)])
        floor = order[rng.integers(0, 6)]
        for p in elig:
            put(p, above(floor))
        pool = elig if elig else []
        k = min(len(pool), int(rng.integers(1, 4)))
        for p in (rng.choice(pool, size=k, replace=False) if k else []):
            put(int(p), floor)
        return {"branch": branch, "floor": floor}
    put(pc, ["at_l", "mid", "at_h"][rng.integers(0, 3)])
    floor = ["zero", "below_l", "at_l", "mid"][rng.integers(0, 4)]
    for p in h.lo:
        put(p, above(floor))
    k = min(len(h.lo), int(rng.integers(1, 4)))
    for p in (rng.choice(h.lo, size=k, replace=False) if k else []):
        put(int(p), floor)
    return {"branch": branch, "floor": floor}


# ----------------------------------------------------------- oracle access
def write_score(pool, head, tier_lists: tuple, pos: int, value):
    """Store `value` as the score of the token at `pos` in the oracle's pages."""
    layer, slot, kvh = head
    hi, lo = tier_lists
    row = pool.table[layer, slot, kvh]
    L = pool.table_len
    if pos in hi:
        s = hi.index(pos)
        page, off = row[s // pool.t_hi], pool.hi_off[4] + 4 * (s % pool.t_hi)
    else:
        s = lo.index(pos)
        page, off = row[L - 1 - s // pool.t_lo], pool.lo_off[4] + 4 * (s % pool.t_lo)
    pool.pages[page, off: off + 4] = np.array([value], F32).view(np.uint8)


def read_record(snap, head, tier, slot, t_hi, t_lo):
    row = snap["table"][head]
    L = row.shape[0]
    if tier == pagefmt.HI:
        return pagefmt.read_token(snap["pages"][row[slot // t_hi]], pagefmt.HI, t_hi, slot % t_hi)
    return pagefmt.read_token(snap["pages"][row[L - 1 - slot // t_lo]], pagefmt.LO, t_lo, slot % t_lo)


def same_record(a: dict, b: dict) -> bool:
    return all((np.asarray(a[k]) == np.asarray(b[k])).all() for k in ("kc", "vc", "ks", "kz", "vs", "vz", "pos")) \
        and np.float32(a["score"]).view(np.uint32) == np.float32(b["score"]).view(np.uint32)


# -------------------------------------------------------------------- test
VARIANTS = {
    "updates": dict(updates=True, lo_enabled=1, recent_window=4),
    # thresholds set for each KV head on its own (Compaction policy, extensibility)
    "per_head_thresholds": dict(updates=True, lo_enabled=1, recent_window=4, per_head=((2.0, 0.25), (1.0, 0.6))),
    "no_updates_w1": dict(updates=False, lo_enabled=1, recent_window=1),
    "lo_disabled": dict(updates=True, lo_enabled=0, recent_window=4),
    "close_thresholds": dict(updates=True, lo_enabled=1, recent_window=3, alpha_h=1.0, alpha_l=0.6),
}


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_decode_step_matches_simulator(variant):
    v = dict(VARIANTS[variant])
    updates = v.pop("updates")
    per_head = v.pop("per_head", None)
    cfg = dict(n_layers=1, n_kv_heads=2, group_size=1, head_dim=128, page_bytes=4096, n_pages=900,
               max_requests=4, max_seq_len=400, tokens_per_hi_page=4, tokens_per_lo_page=8, lo_enabled=1,
               alpha_h=2.0, alpha_l=0.25, recent_window=4, obs_window=32, prompt_grant_slack=1,
               reclaim_in_decode=1)
    cfg.update(v)
    W, lo_enabled = cfg["recent_window"], bool(cfg["lo_enabled"])
    H = cfg["n_kv_heads"]
    slots, lens = [0, 1, 3], [40, 2, 70]
    n_tok = sum(lens)
    pool = oracle.Pool(cfg)
    alphas = [(cfg["alpha_h"], cfg["alpha_l"])] * H
    if per_head is not None:
        alphas = list(per_head)
        assert pool.set_thresholds(0, [a for a, _ in alphas], [b for _, b in alphas]) == 0
    k = workloads.random_fp16((n_tok, H, 128), 5)
    vv = workloads.random_fp16((n_tok, H, 128), 6)
    assert pool.prompt(0, slots, lens, k, vv, scores_in=workloads.given_scores(n_tok, H, seed=7)) == 0
    rng = np.random.default_rng(zlib.crc32(variant.encode()))
    # the simulator starts from the oracle's prompt state (the prompt step has pins of its own)
    snap = pool.snapshot()
    sim, N = {}, {s: n0 for s, n0 in zip(slots, lens)}
    for s, n0 in zip(slots, lens):
        for kvh in range(H):
            hd = (0, s, kvh)
            hp, lp = pagefmt.segment_values(snap, hd, pool.t_hi, pool.t_lo, 5, np.int32)
            cnt = snap["head_counts"][hd]
            h = SimHead(hi=[int(x) for x in hp], lo=[int(x) for x in lp], php=int(cnt[2]), plp=int(cnt[3]))
            for p in h.hi + h.lo:
                h.seen[p] = observation_count(p, n0)
            sim[(s, kvh)] = h
    branches = {}
    for step in range(60):
        # crafted scores, written into the oracle's pages
        for s in slots:
            n = N[s] + 1
            for kvh in range(H):
                th_h, th_l = F32(alphas[kvh][0]) / F32(n), F32(alphas[kvh][1]) / F32(n)
                h = sim[(s, kvh)]
                info = design_scores(h, n, W, th_h, th_l, lo_enabled, rng)
                b = (info.get("branch"), info.get("floor"))
                branches[b] = branches.get(b, 0) + 1
                for p in h.hi + h.lo:
                    write_score(pool, (0, s, kvh), (h.hi, h.lo), p, h.score[p])
        before = pool.snapshot()
        start = int(before["pointers"][0])
        # prediction
        kn = workloads.random_fp16((len(slots), H, 128), 1000 + step)
        vn = workloads.random_fp16((len(slots), H, 128), 2000 + step)
        pred = {}
        aoff = 0
        for i, s in enumerate(slots):
            n = N[s] + 1
            for kvh in range(H):
                th_h, th_l = F32(alphas[kvh][0]) / F32(n), F32(alphas[kvh][1]) / F32(n)
                h = sim[(s, kvh)]
                old_hi, old_lo = list(h.hi), list(h.lo)
                demoted = sim_step(h, n, W, th_h, th_l, lo_enabled)
                need_h, need_l = -(-len(h.hi) // pool.t_hi), -(-len(h.lo) // pool.t_lo)
                new_h, new_l = max(0, need_h - h.php), max(0, need_l - h.plp)
                ids_h = [int(before["free_list"][(start + aoff + x) % cfg["n_pages"]]) for x in range(new_h)]
                aoff += new_h
                ids_l = [int(before["free_list"][(start + aoff + x) % cfg["n_pages"]]) for x in range(new_l)]
                aoff += new_l
                pred[(s, kvh)] = (old_hi, old_lo, demoted, ids_h, ids_l, i)
        assert pool.decode(0, slots, kn, vn) == 0
        after = pool.snapshot()
        assert int(after["pointers"][0]) == start + aoff
        for s in slots:
            N[s] += 1
            assert after["req_state"][0, s, 2] == N[s]
        for (s, kvh), (old_hi, old_lo, demoted, ids_h, ids_l, i) in pred.items():
            h = sim[(s, kvh)]
            hd = (0, s, kvh)
            ctx = f"step {step} slot {s} kvh {kvh}"
            hp, lp = pagefmt.segment_values(after, hd, pool.t_hi, pool.t_lo, 5, np.int32)
            assert hp.tolist() == h.hi, (ctx, "hi slots", hp.tolist(), h.hi)
            assert lp.tolist() == h.lo, (ctx, "lo slots", lp.tolist(), h.lo)
            hs, ls = pagefmt.segment_values(after, hd, pool.t_hi, pool.t_lo, 4, np.float32)
            assert hs.tolist() == [float(h.score[p]) for p in h.hi], ctx
            assert ls.tolist() == [float(h.score[p]) for p in h.lo], ctx
            row, L = after["table"][hd], pool.table_len
            cnt = after["head_counts"][hd]
            assert [int(x) for x in row[h.php:h.php + len(ids_h)]] == ids_h, ctx
            assert [int(row[L - 1 - (h.plp + x)]) for x in range(len(ids_l))] == ids_l, ctx
            h.php += len(ids_h)
            h.plp += len(ids_l)
            assert tuple(int(x) for x in cnt) == (len(h.hi), len(h.lo), h.php, h.plp), ctx
            # codes of every slot whose content changed
            for tier, lst, old in ((pagefmt.HI, h.hi, old_hi), (pagefmt.LO, h.lo, old_lo)):
                for x, p in enumerate(lst):
                    if x < len(old) and old[x] == p:
                        continue
                    got = read_record(after, hd, tier, x, pool.t_hi, pool.t_lo)
                    if p == N[s] - 1:
                        kc, ks, kz = np_quantize(kn[i, kvh].astype(F32), 8)
                        vc, vs, vz = np_quantize(vn[i, kvh].astype(F32), 4)
                        want = dict(kc=kc, vc=vc, ks=ks, kz=kz, vs=vs, vz=vz, score=0.0, pos=p)
                    elif p in demoted:
                        src = read_record(before, hd, pagefmt.HI, old_hi.index(p), pool.t_hi, pool.t_lo)
                        kc, ks, kz = np_quantize(np_dequant(src["kc"], src["ks"], src["kz"]), 4)
                        vc, vs, vz = np_quantize(np_dequant(src["vc"], src["vs"], src["vz"]), 2)
                        want = dict(kc=kc, vc=vc, ks=ks, kz=kz, vs=vs, vz=vz, score=src["score"], pos=p)
                    else:
                        want = read_record(before, hd, tier, old.index(p), pool.t_hi, pool.t_lo)
                    assert same_record(got, want), (ctx, "slot content", tier, x, p)
        pagefmt.check_invariants(after, pool.t_hi, pool.t_lo, cfg["n_pages"])
        if updates:
            for s in slots:
                pool.req_state[0, s, 3] += 1
                for kvh in range(H):
                    h = sim[(s, kvh)]
                    for p in h.hi + h.lo:
                        h.seen[p] += 1
    # every branch of the flow was reached, with several victim levels each
    got = {b for b, _ in branches}
    assert "prune" in got and "hi" in got and (not lo_enabled or "lo" in got), branches
    assert len({f for b, f in branches if b == "hi"}) >= 4, branches


# ------------------------------------------------------- planted mistakes
MUTANTS = {
    "victim_by_argmax": ("a[x].imp < a[best].imp", "a[x].imp > a[best].imp"),
    "tie_to_largest_position": ("a[x].pos < a[best].pos", "a[x].pos > a[best].pos"),
    "hi_threshold_inclusive": ("if (imp > th_h) return TIER_HI;", "if (imp >= th_h) return TIER_HI;"),
    "lo_threshold_exclusive": ("if (imp >= th_l) return TIER_LO;", "if (imp > th_l) return TIER_LO;"),
    "count_off_by_one": ("+ updates - (j >= n0 ? j - n0 : 0)", "+ updates + 1 - (j >= n0 ? j - n0 : 0)"),
    "victim_moved_within_its_level": ("if (tier_rank(cv) < tier_rank(vt)) {", "if (tier_rank(cv) <= tier_rank(vt)) {"),
    "victim_never_moved": ("if (tier_rank(cv) < tier_rank(vt)) {", "if (0) {"),
    "window_ignored": ("argmin_imp(a, q->n[vt], vt == TIER_HI ? n - c->window : 0x7fffffff)",
                       "argmin_imp(a, q->n[vt], 0x7fffffff)"),
    "demoted_pruned_instead": ("if (cv != TIER_PRUNE) q->a[cv][q->n[cv]++] = t;",
                               "if (0) q->a[cv][q->n[cv]++] = t;"),
    "thresholds_of_head0": ("const float* alpha = p->alpha + 2 * hx;",
                            "const float* alpha = p->alpha + 2 * ((size_t)layer * H);"),
}


@pytest.mark.slow
def test_planted_mistakes_are_caught():
    """Each planted mistake, built into a copy of the oracle on the CPU, makes
    the simulator test fail; the unchanged copy passes."""
    src = open(os.path.join(ROOT, "oracle", "dkv_oracle.c")).read()
    with tempfile.TemporaryDirectory() as tmp:
        def run(name, text):
            c_path = os.path.join(tmp, f"{name}.c")
            so_path = os.path.join(tmp, f"{name}.so")
            open(c_path, "w").write(text)
            subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                            "-o", so_path, c_path, "-lm"], check=True)
            env = dict(os.environ, DKV_ORACLE_LIB=so_path)
            r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                                os.path.join(HERE, "test_oracle_decode_sim.py"), "-k", "matches_simulator"],
                               cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
            return r.returncode
        for name, (old, new) in MUTANTS.items():
            assert src.count(old) == 1, f"mutation site of {name} not found once in the oracle"
        jobs = [("unchanged", src)] + [(name, src.replace(old, new)) for name, (old, new) in MUTANTS.items()]
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
            rcs = dict(zip([j[0] for j in jobs], ex.map(lambda j: run(*j), jobs)))
        assert rcs.pop("unchanged") == 0
        survived = [name for name, rc in rcs.items() if rc == 0]
        assert not survived, f"planted mistakes not caught: {survived}"

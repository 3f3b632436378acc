"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs. Integer and page state bit-exact; scores and attention
within stated tolerances."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads
from tests import parity
from tests.gpu_pool import GPool, stored, tiers_of

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# Attention: |gpu - ref| <= ATOL + RTOL |ref| elementwise (fp64 reference over
# the same dequantised values).
ATT_ATOL, ATT_RTOL = 1e-3, 2e-3
# Scores: fp32 tensor-core logits and exp2 against fp64: relative error of a
# few fp32 roundings per term, summed over at most 32 observation queries.
SC_ATOL, SC_RTOL = 1e-6, 5e-5
# Tie band, from the score tolerance: a GPU score within SC_ATOL + SC_RTOL*S of
# the fp64 score gives an importance within that error over c, plus the fp32
# roundings of I and of alpha/N (2^-22 relative); only a token whose fp64
# importance lies that close to a threshold may land on the other side.
ROUND_REL = 2.0 ** -22


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiated_kv_cache_gb300 as dkv
    dkv.build.build()
    dkv.load()


def cfg_of(**over):
    c = dict(n_layers=1, n_kv_heads=2, group_size=4, head_dim=128, page_bytes=4096, n_pages=512,
             max_requests=6, max_seq_len=1200, tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=1,
             alpha_h=2.0, alpha_l=0.25, recent_window=64, obs_window=32, prompt_grant_slack=1,
             reclaim_in_decode=1)
    c.update(over)
    return c


def both(cfg):
    return GPool(cfg), oracle.Pool(cfg)


def assert_same(gp, op, **kw):
    parity.compare_states(gp.snapshot(), op.snapshot(), gp.t_hi, gp.t_lo, gp.cfg["n_pages"],
                          gp.cfg["page_bytes"], **kw)


# ------------------------------------------------------------------ Figure 6
def test_figure6_on_gpu():
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fig6_prompt_workflow.json")))
    cfg = cfg_of(tokens_per_hi_page=2, tokens_per_lo_page=4, prompt_grant_slack=0, recent_window=0,
                 n_pages=16, max_requests=1, max_seq_len=8)
    tiers = {0: "HLLPHLPL", 1: "HHLHLPHP"}
    imp = {"H": 1.0, "L": 0.1, "P": 0.001}
    S = np.array([[imp[tiers[h][j]] * min(32, 8 - j) for h in (0, 1)] for j in range(8)], np.float32)
    k = workloads.random_fp16((8, 2, 128), 1)
    v = workloads.random_fp16((8, 2, 128), 2)
    gp, op = both(cfg)
    with gp:
        gp.prompt(0, [0], [8], k, v, scores_in=S)
        assert op.prompt(0, [0], [8], k, v, scores_in=S) == 0
        snap = gp.snapshot()
        # the page's example starts with pages 0-4 allocated; here the list starts at 0,
        # so every page ID is the figure's minus 5
        sh = gold["config"]["list_start_before"]
        L = gp.table_len
        for h, name in ((0, "A"), (1, "B")):
            row = snap["table"][0, 0, h]
            hi = gold["expected"]["hi_pages"][name]; lo = gold["expected"]["lo_pages"][name]
            assert [int(x) + sh for x in row[:len(hi)]] == hi
            assert [int(row[L - 1 - x]) + sh for x in range(len(lo))] == lo
        rec = [int(snap["free_list"][c % 16]) + sh for c in range(16, int(snap["pointers"][1]))]
        assert rec == gold["expected"]["reclaimed_in_order"]
        assert int(snap["pointers"][0]) + sh == gold["expected"]["list_start_after"]
        assert_same(gp, op)


# ---------------------------------------------------- prompt, given scores
@pytest.mark.parametrize("pb", [4096, 3584])
@pytest.mark.parametrize("G,H,lens", [(4, 2, [512, 700]), (1, 3, [1, 31, 129, 300]), (5, 2, [1029, 64, 65]),
                                      (7, 1, [777]), (8, 2, [256, 257])])
def test_prompt_given_scores_bit_exact(G, H, lens, pb):
    cfg = cfg_of(group_size=G, n_kv_heads=H, n_pages=2048, max_requests=len(lens) + 1, page_bytes=pb)
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 10 + G, scale=2.0)
    v = workloads.random_fp16((n, H, 128), 20 + G)
    S = workloads.given_scores(n, H, seed=G, scale=1.0)
    slots = list(range(1, len(lens) + 1))           # not starting at 0
    gp, op = both(cfg)
    with gp:
        rc, so = gp.prompt(0, slots, lens, k, v, scores_in=S, want_scores=True)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        assert (so == S).all()
        assert_same(gp, op)
        st = gp.status()
        assert st["error"] == 0 and st["hi_tokens"] + st["lo_tokens"] > 0


@pytest.mark.parametrize("over", [dict(lo_enabled=0), dict(alpha_h=math.inf, alpha_l=0.0),
                                  dict(alpha_h=0.0, alpha_l=0.0), dict(recent_window=0),
                                  dict(tokens_per_hi_page=4, tokens_per_lo_page=8, prompt_grant_slack=3)])
def test_prompt_special_configs_bit_exact(over):
    cfg = cfg_of(n_pages=2048, **over)
    lens = [300, 5, 700]
    n = sum(lens)
    k = workloads.random_fp16((n, 2, 128), 1)
    v = workloads.random_fp16((n, 2, 128), 2)
    S = workloads.given_scores(n, 2, seed=3)
    gp, op = both(cfg)
    with gp:
        gp.prompt(0, [0, 1, 2], lens, k, v, scores_in=S)
        assert op.prompt(0, [0, 1, 2], lens, k, v, scores_in=S) == 0
        assert_same(gp, op)


# ------------------------------------------------- prompt, computed scores
def _tie_tokens(S64, lens, H, alpha_h, alpha_l, window, lo_enabled):
    ties = np.zeros(S64.shape, bool)
    t0 = 0
    for n0 in lens:
        j = np.arange(n0)
        c = np.minimum(32, n0 - j)[:, None].astype(np.float64)
        I = S64[t0:t0 + n0] / c * n0
        err = (SC_RTOL + ROUND_REL) * I + SC_ATOL / c * n0
        near = np.zeros_like(I, bool)
        for a in ([alpha_h, alpha_l] if lo_enabled else [alpha_l]):
            if np.isfinite(a) and a > 0:
                near |= np.abs(I - a) <= err + ROUND_REL * a
        near[j >= n0 - window] = False
        ties[t0:t0 + n0] = near
        t0 += n0
    return ties


def _inputs(name, reqs, max_len, G_override=None):
    """Workload inputs for a few requests, prompts cut to max_len tokens
    (the observation queries stay those of the generated prompt)."""
    if name == "random8":
        rng_k = workloads.random_fp16((1700, 2, 128), 77, scale=1.5)
        return dict(k=rng_k, v=workloads.random_fp16((1700, 2, 128), 78),
                    q_obs=workloads.random_fp16((2, 32, 16, 128), 79), lens=np.array([700, 1000], np.int32)), 2
    inp = workloads.prompt_inputs(name, 0, requests=reqs)
    H = workloads.WORKLOADS[name].n_kv_heads
    lens = [int(x) for x in inp["lens"]]
    if max(lens) > max_len:
        ks, vs, t0 = [], [], 0
        for n0 in lens:
            m = min(n0, max_len)
            ks.append(inp["k"][t0:t0 + m]); vs.append(inp["v"][t0:t0 + m])
            t0 += n0
        inp["k"], inp["v"] = np.concatenate(ks), np.concatenate(vs)
        inp["lens"] = np.minimum(inp["lens"], max_len)
    return inp, H


@pytest.mark.parametrize("name,G,reqs", [("tiny", 4, None), ("qwq32b", 5, [0, 1]), ("qwen7b", 7, [0]),
                                         ("random8", 8, None)])
def test_prompt_computed_scores(name, G, reqs):
    inp, H = _inputs(name, reqs, 3000)
    lens = [int(x) for x in inp["lens"]]
    lo_enabled = workloads.WORKLOADS[name].lo_enabled if name in workloads.WORKLOADS else 1
    cfg = cfg_of(n_kv_heads=H, group_size=G, n_pages=4096, max_requests=len(lens), max_seq_len=max(lens) + 8,
                 lo_enabled=lo_enabled)
    gp = GPool(cfg)
    op = oracle.Pool(cfg)
    slots = list(range(len(lens)))
    with gp:
        rc, so = gp.prompt(0, slots, lens, inp["k"], inp["v"], inp["q_obs"], want_scores=True)
        S64 = np.zeros((sum(lens), H))
        t0 = 0
        for i, n0 in enumerate(lens):
            for h in range(H):
                S64[t0:t0 + n0, h] = oracle.unit_scores(inp["k"][t0:t0 + n0, h],
                                                        inp["q_obs"][i][:, h * G:(h + 1) * G])
            t0 += n0
        ok, worst = parity.within(so.astype(np.float64), S64, SC_ATOL, SC_RTOL)
        rel = np.abs(so - S64) / np.maximum(S64, 1e-30)
        print(f"{name}: score max rel err {rel.max():.3e}, tolerance excess {worst:.3e}")
        assert ok, worst
        ties = _tie_tokens(S64, lens, H, cfg["alpha_h"], cfg["alpha_l"], cfg["recent_window"], cfg["lo_enabled"])
        assert op.prompt(0, slots, lens, inp["k"], inp["v"], inp["q_obs"]) == 0
        gs, os_ = gp.snapshot(), op.snapshot()
        t0 = 0
        clean = []
        for i, n0 in enumerate(lens):
            for h in range(H):
                tg = tiers_of(gs, (0, i, h), n0, gp.t_hi, gp.t_lo)
                to = tiers_of(os_, (0, i, h), n0, gp.t_hi, gp.t_lo)
                tie = ties[t0:t0 + n0, h]
                assert (tg[~tie] == to[~tie]).all(), f"tier differs outside the tie band (req {i}, head {h})"
                if (tg == to).all():
                    clean.append((0, i, h))
            t0 += n0
        print(f"{name}: {int(ties.sum())} tokens in the tie band; {len(clean)}/{len(lens) * H} heads identical")
        # heads whose tiers agree: identical pages up to the score words (fp32 vs fp64 sums)
        parity.compare_states(gs, os_, gp.t_hi, gp.t_lo, cfg["n_pages"], cfg["page_bytes"], heads=clean,
                              scores=False)
        if len(clean) == len(lens) * H:
            parity.compare_states(gs, os_, gp.t_hi, gp.t_lo, cfg["n_pages"], cfg["page_bytes"], scores=False)


# --------------------------------------------------------------- decode
@pytest.mark.parametrize("over", [dict(), dict(alpha_h=1.0, alpha_l=0.6), dict(lo_enabled=0, alpha_l=0.5),
                                  dict(tokens_per_hi_page=2, tokens_per_lo_page=4, recent_window=3),
                                  dict(reclaim_in_decode=0, alpha_h=4.0, alpha_l=1.0, recent_window=8),
                                  dict(page_bytes=3584), dict(page_bytes=3584, alpha_h=1.0, alpha_l=0.6)])
def test_decode_steps_bit_exact(over):
    cfg = cfg_of(max_seq_len=1000, n_pages=4096, **over)
    lens = [200, 333, 70]
    n = sum(lens)
    H = cfg["n_kv_heads"]
    k = workloads.random_fp16((n, H, 128), 7)
    v = workloads.random_fp16((n, H, 128), 8)
    S = workloads.given_scores(n, H, seed=9)
    slots = [0, 2, 4]
    gp, op = both(cfg)
    with gp:
        gp.prompt(0, slots, lens, k, v, scores_in=S)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        for step in range(40):
            kn = workloads.random_fp16((3, H, 128), 100 + step)
            vn = workloads.random_fp16((3, H, 128), 200 + step)
            gp.decode(0, slots, kn, vn)
            assert op.decode(0, slots, kn, vn) == 0
            if step % 8 == 7 or step < 3:
                assert_same(gp, op)
        for s in slots:
            gp.free(s)
            assert op.free_request(s) == 0
        assert_same(gp, op)
        st = gp.status()
        assert st["free_pages"] == cfg["n_pages"] and st["error"] == 0


# ------------------------------------------------------------ attention
@pytest.mark.parametrize("pb", [4096, 3584])
@pytest.mark.parametrize("G,H,lens,steps", [(4, 2, [512, 700], 5), (1, 2, [40, 1], 3), (5, 3, [1030, 17], 2),
                                            (7, 1, [2000], 1), (8, 2, [300, 301], 4)])
def test_decode_attention_parity(G, H, lens, steps, pb):
    cfg = cfg_of(group_size=G, n_kv_heads=H, n_pages=4096, max_seq_len=2100, max_requests=len(lens), page_bytes=pb)
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 30, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 31)
    S = workloads.given_scores(n, H, seed=32)
    slots = list(range(len(lens)))
    gp, op = both(cfg)
    with gp:
        gp.prompt(0, slots, lens, k, v, scores_in=S)
        op.prompt(0, slots, lens, k, v, scores_in=S)
        for step in range(steps):
            kn = workloads.random_fp16((len(lens), H, 128), 300 + step)
            vn = workloads.random_fp16((len(lens), H, 128), 400 + step)
            gp.decode(0, slots, kn, vn)
            op.decode(0, slots, kn, vn)
            q = workloads.random_fp16((len(lens), H * G, 128), 500 + step, scale=2.0)
            out = gp.attention(0, slots, q)
            rc, ref = op.attention(0, slots, q)
            ok, worst = parity.within(out.astype(np.float64), ref, ATT_ATOL, ATT_RTOL)
            ratio = (np.abs(out - ref) / (ATT_ATOL + ATT_RTOL * np.abs(ref))).max()
            print(f"G={G}: attention max abs err {np.abs(out - ref).max():.3e}, max err/tolerance {ratio:.3f}")
            assert ok, worst
        assert_same(gp, op)


def test_attention_large_pages_four_warp_ctas():
    """Pages of 32 hi / 64 lo tokens (8 KB): the paged kernel's rings of 16
    warps do not fit in shared memory, so it runs as four CTAs of 4 warps per
    SM; outputs with and without score updates against the oracle."""
    G, H, lens = 4, 2, [900, 333]
    cfg = cfg_of(group_size=G, n_kv_heads=H, n_pages=1024, max_seq_len=1000, max_requests=2, page_bytes=8192,
                 tokens_per_hi_page=32, tokens_per_lo_page=64)
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 60, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 61)
    S = workloads.given_scores(n, H, seed=62)
    gp, op = both(cfg)
    with gp:
        assert (gp.t_hi, gp.t_lo) == (32, 64)
        gp.prompt(0, [0, 1], lens, k, v, scores_in=S)
        op.prompt(0, [0, 1], lens, k, v, scores_in=S)
        for step, update in enumerate([False, True, True]):
            q = workloads.random_fp16((2, H * G, 128), 650 + step, scale=2.0)
            out = gp.attention(0, [0, 1], q, update=update)
            rc, ref = op.attention(0, [0, 1], q, update_scores=update)
            ok, worst = parity.within(out.astype(np.float64), ref, ATT_ATOL, ATT_RTOL)
            assert ok, (step, worst)
        gs, os_ = gp.snapshot(), op.snapshot()
        for i in range(2):
            for h in range(H):
                for a, b in zip(stored(gs, (0, i, h), gp.t_hi, gp.t_lo, 4, np.float32),
                                stored(os_, (0, i, h), gp.t_hi, gp.t_lo, 4, np.float32)):
                    ok, worst = parity.within(a.astype(np.float64), b.astype(np.float64), 1e-6, 1e-4)
                    assert ok, worst


@pytest.mark.parametrize("pb", [4096, 3584])
def test_attention_score_update(pb):
    cfg = cfg_of(group_size=4, n_kv_heads=2, n_pages=2048, max_requests=2, page_bytes=pb)
    lens = [600, 257]
    n = sum(lens)
    k = workloads.random_fp16((n, 2, 128), 40, scale=1.5)
    v = workloads.random_fp16((n, 2, 128), 41)
    S = workloads.given_scores(n, 2, seed=42)
    gp, op = both(cfg)
    with gp:
        gp.prompt(0, [0, 1], lens, k, v, scores_in=S)
        op.prompt(0, [0, 1], lens, k, v, scores_in=S)
        for step in range(3):
            q = workloads.random_fp16((2, 8, 128), 600 + step, scale=2.0)
            gp.attention(0, [0, 1], q, update=True)
            op.attention(0, [0, 1], q, update_scores=True)
        gs, os_ = gp.snapshot(), op.snapshot()
        assert (gs["req_state"] == os_["req_state"]).all()
        for i in range(2):
            for h in range(2):
                for a, b in zip(stored(gs, (0, i, h), gp.t_hi, gp.t_lo, 4, np.float32),
                                stored(os_, (0, i, h), gp.t_hi, gp.t_lo, 4, np.float32)):
                    ok, worst = parity.within(a.astype(np.float64), b.astype(np.float64), 1e-6, 1e-4)
                    assert ok, worst


# -------------------------------------------------------------- errors
def test_errors_are_transactional_and_sticky():
    cfg = cfg_of(n_pages=40)
    lens = [500]
    k = workloads.random_fp16((500, 2, 128), 1)
    S = workloads.given_scores(500, 2, seed=1)
    gp, op = both(cfg)
    with gp:
        before = gp.snapshot()
        gp.prompt(0, [0], lens, k, k, scores_in=S)          # needs 2 x 29 pages > 40
        st = gp.status()
        assert st["error"] == -4 and st["free_pages"] == 40
        after = gp.snapshot()
        for key in ("free_list", "table", "head_counts", "req_state", "pointers"):
            assert (before[key] == after[key]).all(), key
        # sticky: a call that would fit is a no-op until the error is cleared
        gp.prompt(0, [1], [10], k[:10], k[:10], scores_in=S[:10])
        assert gp.status()["hi_tokens"] == 0
        import differentiated_kv_cache_gb300 as dkv
        dkv.dkv_pool_clear_error(gp.h)
        gp.prompt(0, [1], [10], k[:10], k[:10], scores_in=S[:10])
        assert op.prompt(0, [1], [10], k[:10], k[:10], scores_in=S[:10]) == 0
        assert gp.status()["error"] == 0
        assert_same(gp, op)
        # host-side state errors return at once
        assert gp.decode(0, [0], k[:1], k[:1], check=False) == dkv.DKV_ERR_STATE
        assert gp.free(3, check=False) == dkv.DKV_ERR_STATE
        assert gp.prompt(0, [1], [10], k[:10], k[:10], scores_in=S[:10], check=False) == dkv.DKV_ERR_STATE


def test_grant_short_with_zero_slack():
    cfg = cfg_of(tokens_per_hi_page=2, tokens_per_lo_page=4, prompt_grant_slack=0, recent_window=0,
                 max_seq_len=8, n_pages=16)
    S = np.zeros((2, 2), np.float32); S[0] = 10.0; S[1] = 0.2
    k = workloads.random_fp16((2, 2, 128), 3)
    with GPool(cfg) as gp:
        before = gp.snapshot()
        gp.prompt(0, [0], [2], k, k, scores_in=S)
        assert gp.status()["error"] == -5
        after = gp.snapshot()
        for key in ("free_list", "table", "head_counts", "req_state", "pointers"):
            assert (before[key] == after[key]).all(), key


def test_argument_errors_queue_nothing_and_length_limit():
    """Calls the host refuses (empty calls, a slot given twice or out of
    range, prompts of 0 tokens or longer than max_seq_len, a layer out of
    range, a misaligned tensor, arguments of the other mode, inactive slots)
    return their code at once, change nothing and latch nothing. A request
    grown to exactly max_seq_len by generation steps matches the oracle bit
    for bit, its next step is refused on both sides as a whole (the other
    request of the call does not step either), and attention over it stays
    within the element-wise bound."""
    import differentiated_kv_cache_gb300 as dkv
    L = 300
    cfg = cfg_of(max_seq_len=L, n_pages=1024)
    H, G = cfg["n_kv_heads"], cfg["group_size"]
    lens, slots = [L - 3, 40, L], [5, 0, 3]
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 31)
    v = workloads.random_fp16((n, H, 128), 32)
    S = workloads.given_scores(n, H, seed=33)
    E_ARG, E_STATE = dkv.DKV_ERR_ARG, dkv.DKV_ERR_STATE
    P, D = dkv.DKV_PROMPT, dkv.DKV_DECODE
    gp, op = both(cfg)
    with gp:
        kd, vd, sd = gp.dev(k), gp.dev(v), gp.dev(S.astype(np.float32))
        kn, vn = gp.dev(k[:3]), gp.dev(v[:3])
        q = gp.dev(workloads.random_fp16((3, H * G, 128), 34))
        out = torch.zeros((3, H * G, 128), dtype=torch.float32, device="cuda")
        before = gp.snapshot()

        def refused(rc, want, what):
            assert rc == want, (what, rc)

        for layer, sl, ln, what in [(0, [], [], "empty call"), (0, [1, 1], [10, 10], "slot twice"),
                                    (0, [6], [10], "slot = max_requests"), (0, [-1], [10], "negative slot"),
                                    (0, [1], [0], "empty prompt"), (0, [1], [L + 1], "beyond max_seq_len"),
                                    (1, [1], [10], "layer out of range")]:
            refused(dkv.dkv_compact_step(gp.h, layer, P, sl, ln, kd, vd, None, sd, check=False), E_ARG, what)
        refused(dkv.dkv_compact_step(gp.h, 0, P, [1], [10], kd.reshape(-1)[1:], vd, None, sd, check=False),
                E_ARG, "keys 2 bytes past a 16-byte boundary")
        refused(dkv.dkv_compact_step(gp.h, 0, P, [1], [10], kd, vd, None, None, check=False), E_ARG,
                "prompt without observation queries or scores")
        refused(dkv.dkv_compact_step(gp.h, 0, 7, [1], [10], kd, vd, None, sd, check=False), E_ARG, "mode 7")
        refused(dkv.dkv_compact_step(gp.h, 0, D, [1], [10], kn, vn, check=False), E_ARG, "lengths in DECODE")
        refused(dkv.dkv_compact_step(gp.h, 0, D, [], None, kn, vn, check=False), E_ARG, "empty generation step")
        refused(dkv.dkv_compact_step(gp.h, 0, D, [1], None, kn, vn, check=False), E_STATE, "inactive slot")
        refused(dkv.dkv_decode_attention(gp.h, 0, [], q, out, True, check=False), E_ARG, "empty attention call")
        refused(dkv.dkv_decode_attention(gp.h, 0, [2], q, out, True, check=False), E_STATE, "attention, inactive")
        refused(dkv.dkv_free_request(gp.h, 6, check=False), E_ARG, "free, slot out of range")
        refused(dkv.dkv_free_request(gp.h, 2, check=False), E_STATE, "free, inactive slot")
        torch.cuda.synchronize()
        after = gp.snapshot()
        for key in ("free_list", "table", "head_counts", "req_state", "pointers"):
            assert (before[key] == after[key]).all(), key
        assert gp.status()["error"] == 0

        # a request at max_seq_len - 3, another at max_seq_len itself
        gp.prompt(0, slots, lens, k, v, scores_in=S)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        assert_same(gp, op)
        assert gp.decode(0, [3], k[:1], v[:1], check=False) == E_ARG
        assert op.decode(0, [3], k[:1], v[:1]) == E_ARG
        for step in range(4):
            kn = workloads.random_fp16((2, H, 128), 40 + step)
            vn = workloads.random_fp16((2, H, 128), 50 + step)
            want = 0 if step < 3 else E_ARG
            assert gp.decode(0, [5, 0], kn, vn, check=False) == want
            assert op.decode(0, [5, 0], kn, vn) == want
            assert_same(gp, op)
        assert gp.status()["error"] == 0
        qa = workloads.random_fp16((3, H * G, 128), 35, scale=2.0)
        got = gp.attention(0, slots, qa, update=False)
        rc, ref = op.attention(0, slots, qa, update_scores=False)
        assert rc == 0
        ok, worst = parity.within(got.astype(np.float64), ref, ATT_ATOL, ATT_RTOL)
        assert ok, worst
        for s in slots:
            gp.free(s)
            assert op.free_request(s) == 0
        assert_same(gp, op)
        assert gp.status()["free_pages"] == cfg["n_pages"]


def test_largest_call():
    """The most requests one call takes (1024, so 2048 heads: the single-CTA
    page allocation of a generation step then holds two heads a thread):
    prompt, three generation steps and request completion bit-exact, the
    attention call within the element-wise bound; a call of 1025 requests
    is refused on the host."""
    import differentiated_kv_cache_gb300 as dkv
    R = 1024
    cfg = cfg_of(max_requests=R, max_seq_len=64, n_pages=12000)
    H, G = cfg["n_kv_heads"], cfg["group_size"]
    lens = [int(x) for x in np.random.default_rng(61).integers(1, 49, R)]
    slots = [int(s) for s in np.random.default_rng(62).permutation(R)]
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 63)
    v = workloads.random_fp16((n, H, 128), 64)
    S = workloads.given_scores(n, H, seed=65)
    gp, op = both(cfg)
    with gp:
        gp.prompt(0, slots, lens, k, v, scores_in=S)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        assert_same(gp, op)
        for step in range(3):
            kn = workloads.random_fp16((R, H, 128), 70 + step)
            vn = workloads.random_fp16((R, H, 128), 80 + step)
            gp.decode(0, slots, kn, vn)
            assert op.decode(0, slots, kn, vn) == 0
            assert_same(gp, op)
        q = workloads.random_fp16((R, H * G, 128), 66, scale=2.0)
        got = gp.attention(0, slots, q, update=False)
        rc, ref = op.attention(0, slots, q, update_scores=False)
        assert rc == 0
        ok, worst = parity.within(got.astype(np.float64), ref, ATT_ATOL, ATT_RTOL)
        assert ok, worst
        for s in slots[:R // 2]:
            gp.free(s)
            assert op.free_request(s) == 0
        assert_same(gp, op)
        assert gp.status()["error"] == 0
    with GPool(cfg_of(max_requests=R + 1, max_seq_len=64, n_pages=64)) as big:
        kd = big.dev(workloads.random_fp16((R + 1, H, 128), 67))
        q = big.dev(workloads.random_fp16((R + 1, H * G, 128), 68))
        out = torch.zeros((R + 1, H * G, 128), dtype=torch.float32, device="cuda")
        assert dkv.dkv_compact_step(big.h, 0, dkv.DKV_PROMPT, list(range(R + 1)), [1] * (R + 1), kd, kd, None,
                                    big.dev(np.ones((R + 1, H), np.float32)), check=False) == dkv.DKV_ERR_ARG
        assert dkv.dkv_decode_attention(big.h, 0, list(range(R + 1)), q, out, False, check=False) == \
            dkv.DKV_ERR_ARG


def test_attention_on_workload_with_outliers():
    """The tiny workload itself (outlier channels x8, scores computed from the
    observation queries), a few decode steps with score updates: attention
    against the oracle's fp64 attention over its own pages."""
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.prompt_inputs("tiny", 0)
    lens = [int(x) for x in inp["lens"]]
    cfg = w.pool_config()
    gp, op = both(cfg)
    with gp:
        gp.prompt(0, [0, 1], lens, inp["k"], inp["v"], inp["q_obs"])
        op.prompt(0, [0, 1], lens, inp["k"], inp["v"], inp["q_obs"])
        gs, os_ = gp.snapshot(), op.snapshot()
        if not ((gs["head_counts"] == os_["head_counts"]).all() and (gs["table"] == os_["table"]).all()):
            pytest.skip("a tie-band token put the two pools on different tiers")
        worst_ratio = 0.0
        for step in range(4):
            d = workloads.decode_inputs("tiny", step)
            gp.decode(0, [0, 1], d["k"], d["v"])
            op.decode(0, [0, 1], d["k"], d["v"])
            out = gp.attention(0, [0, 1], d["q"], update=False)
            rc, ref = op.attention(0, [0, 1], d["q"], update_scores=False)
            ratio = (np.abs(out - ref) / (ATT_ATOL + ATT_RTOL * np.abs(ref))).max()
            worst_ratio = max(worst_ratio, ratio)
        print(f"tiny workload: attention max err/tolerance {worst_ratio:.3f}")
        assert worst_ratio <= 1.0


# ------------------------------------------------- per-head thresholds
def test_per_head_thresholds_bit_exact():
    """Thresholds for each KV head (DiffKV compaction policy, extensibility),
    two layers with different pairs, changed between generation steps: the
    prompt with caller scores, then steps of (compaction, attention with
    score update) with the oracle taken over from the GPU state before each
    step; every state bit-exact."""
    import differentiated_kv_cache_gb300 as dkv
    from tests.gpu_pool import load_into
    H, G = 4, 4
    cfg = cfg_of(n_layers=2, n_kv_heads=H, group_size=G, n_pages=4096, max_seq_len=1400, page_bytes=3584,
                 recent_window=16)
    lens, slots = [900, 400], [1, 0]
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 51, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 52)
    S = workloads.given_scores(n, H, seed=53, scale=0.2)
    pairs = {0: ([2.0, 0.5, 4.0, 1.0], [0.25, 0.05, 1.0, 0.9]), 1: ([1.0, 1.0, 8.0, 0.3], [0.6, 0.0, 0.5, 0.3])}
    gp, op = both(cfg)
    with gp:
        for layer, (ah, al) in pairs.items():
            dkv.dkv_pool_set_thresholds(gp.h, layer, ah, al)
            assert op.set_thresholds(layer, ah, al) == 0
        for layer in (0, 1):
            gp.prompt(layer, slots, lens, k, v, scores_in=S)
            assert op.prompt(layer, slots, lens, k, v, scores_in=S) == 0
        assert_same(gp, op)
        for step in range(30):
            if step == 15:                       # new pairs for layer 0 mid-run
                ah, al = [0.5, 3.0, 1.0, 2.0], [0.1, 0.5, 0.5, 0.0]
                dkv.dkv_pool_set_thresholds(gp.h, 0, ah, al)
                assert op.set_thresholds(0, ah, al) == 0
            layer = step % 2
            kn = workloads.random_fp16((2, H, 128), 5000 + step)
            vn = workloads.random_fp16((2, H, 128), 6000 + step)
            load_into(op, gp.snapshot())
            gp.decode(layer, slots, kn, vn)
            assert op.decode(layer, slots, kn, vn) == 0
            assert_same(gp, op)
            q = workloads.random_fp16((2, H * G, 128), 7000 + step, scale=2.0)
            gp.attention(layer, slots, q, update=True)
        assert gp.status()["error"] == 0
        assert dkv.dkv_pool_set_thresholds(gp.h, 0, [float("nan")] * H, [0.1] * H, check=False) == dkv.DKV_ERR_ARG
        assert dkv.dkv_pool_set_thresholds(gp.h, 2, [1.0] * H, [0.1] * H, check=False) == dkv.DKV_ERR_ARG

"""Pins of the CPU oracle to facts outside itself: numpy/scipy routines, the
DiffKV page's Figure 6 worked example, closed forms, special cases and the
memory-management invariants. None of these re-types the oracle's formulas."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import workloads
from tests import pagefmt

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_cfg(**over):
    cfg = dict(n_layers=1, n_kv_heads=2, group_size=4, head_dim=128, page_bytes=4096, n_pages=256,
               max_requests=4, max_seq_len=512, tokens_per_hi_page=0, tokens_per_lo_page=0,
               lo_enabled=1, alpha_h=2.0, alpha_l=0.25, recent_window=64, obs_window=32,
               prompt_grant_slack=1, reclaim_in_decode=1)
    cfg.update(over)
    return cfg


# ---------------------------------------------------------------- fp16 ----
def test_half_conversion_matches_numpy():
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * s for s in (1e-8, 1e-6, 1e-4, 1, 100, 3e4)
    ] + [np.array([0.0, -0.0, 65504, 65519.99, 65520, -65520, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8,
                   1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 2048 + 1, 2048 + 3], np.float32)])
    want = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half_bits(float(x)) for x in xs], np.uint16)
    assert (got == want).all()
    hs = np.arange(0, 65536, 7, dtype=np.uint16)
    hs = hs[(hs & 0x7c00) != 0x7c00]
    back = np.array([oracle.half_bits_to_float(int(h)) for h in hs], np.float32)
    assert (back == hs.view(np.float16).astype(np.float32)).all()


# ---------------------------------------------------------------- codec ---
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codec_exact_on_grid(bits):
    """Values already on a grid z + s*k (s, z binary16, codes 0 and L present)
    come back as exactly those codes, scale and zero, and dequantise exactly."""
    rng = np.random.default_rng(bits)
    L = (1 << bits) - 1
    for s, z in [(2.0 ** -4, -8.0), (0.5, 3.0), (2.0 ** -10, 0.0), (3.0, -100.0)]:
        k = rng.integers(0, L + 1, size=128)
        k[3], k[77] = 0, L
        x = (z + s * k).astype(np.float32)
        codes, sb, zb = oracle.quantize(x, bits)
        assert (codes == k).all()
        assert sb == np.float16(s).view(np.uint16) and zb == np.float16(z).view(np.uint16)
        assert (oracle.dequant(sb, zb, codes) == x).all()


def test_codec_textbook_example():
    codes, sb, zb = oracle.quantize(np.array([0, 1, 2, 3], np.float32), 2)
    assert list(codes) == [0, 1, 2, 3] and sb == 0x3C00 and zb == 0


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codec_round_trip_bound_and_order(bits):
    """|x - x^| <= s/2 + L|s - s_exact| + |z - min| + 4 ulp(max|x|); codes in
    [0, L]; the map x -> code is monotone."""
    rng = np.random.default_rng(10 + bits)
    L = (1 << bits) - 1
    vecs = [rng.standard_normal(128), rng.standard_normal(128) * 1e-3,
            np.where(rng.random(128) < 0.03, 8.0, 1.0) * rng.standard_normal(128),
            np.full(128, 0.7), np.linspace(-65504, 65504, 128), rng.standard_normal(128) * 1e-6]
    for x in vecs:
        x = x.astype(np.float16).astype(np.float32)
        codes, sb, zb = oracle.quantize(x, bits)
        s = float(np.uint16(sb).view(np.float16)); z = float(np.uint16(zb).view(np.float16))
        mn, mx = float(x.min()), float(x.max())
        s_exact = (mx - mn) / L
        xh = oracle.dequant(sb, zb, codes).astype(np.float64)
        ulp = 4 * np.spacing(np.float32(max(abs(mn), abs(mx), 1e-30)))
        bound = 0.5 * s + L * abs(s - s_exact) + abs(z - mn) + ulp
        assert np.abs(x - xh).max() <= bound * (1 + 1e-6)
        assert codes.min() >= 0 and codes.max() <= L
        order = np.argsort(x, kind="stable")
        assert (np.diff(codes[order].astype(int)) >= 0).all()


def test_codec_constant_and_signed_zero():
    codes, sb, zb = oracle.quantize(np.full(128, 1.2345, np.float32), 8)
    assert (codes == 0).all() and sb == 0 and zb == np.float16(1.2345).view(np.uint16)
    x = np.zeros(128, np.float32); x[5] = -0.0; x[9] = 1.0
    _, _, zb = oracle.quantize(x, 4)
    assert zb == 0  # -0 is taken as +0


# ---------------------------------------------------------------- scores --
def _dense_softmax_scores(k, q):
    """Reference for G = 1: S_j = sum over observation rows p >= j of
    softmax(q_p . K^T / sqrt(d))_j, built with scipy's softmax on a dense
    causal logit matrix."""
    n0 = k.shape[0]
    kk = k.astype(np.float64); qq = q[:, 0, :].astype(np.float64)
    S = np.zeros(n0)
    for o in range(32):
        p = n0 - 32 + o
        if p < 0:
            continue
        logits = kk[:p + 1] @ qq[o] / math.sqrt(128)
        S[:p + 1] += scipy.special.softmax(logits)
    return S


@pytest.mark.parametrize("n0", [5, 31, 32, 33, 200])
def test_scores_g1_match_scipy_softmax(n0):
    rng = np.random.default_rng(n0)
    k = (rng.standard_normal((n0, 128)) * 1.5).astype(np.float16)
    q = rng.standard_normal((32, 1, 128)).astype(np.float16)
    S = oracle.unit_scores(k, q)
    np.testing.assert_allclose(S, _dense_softmax_scores(k, q), rtol=1e-12, atol=1e-15)
    assert abs(S.sum() - min(32, n0)) < 1e-9          # every softmax row sums to one


def test_scores_group_max_properties():
    rng = np.random.default_rng(7)
    n0 = 150
    k = rng.standard_normal((n0, 128)).astype(np.float16)
    q1 = rng.standard_normal((32, 1, 128)).astype(np.float16)
    # identical heads in a group: the max equals the single head
    same = oracle.unit_scores(k, np.repeat(q1, 4, axis=1))
    np.testing.assert_allclose(same, oracle.unit_scores(k, q1), rtol=1e-13)
    # distinct heads: bounded by the single-head scores of each head
    q4 = rng.standard_normal((32, 4, 128)).astype(np.float16)
    S4 = oracle.unit_scores(k, q4)
    per = np.stack([oracle.unit_scores(k, q4[:, h:h + 1]) for h in range(4)])
    assert (S4 >= per.max(0) - 1e-12).all() and (S4 <= per.sum(0) + 1e-12).all()
    assert 32 - 1e-9 <= S4.sum() <= 32 * 4 + 1e-9
    # causality: changing observation row o (position p) leaves S_j, j > p, unchanged
    q5 = q4.copy(); q5[10] = rng.standard_normal((4, 128)).astype(np.float16)
    d = oracle.unit_scores(k, q5) - S4
    p = n0 - 32 + 10
    assert np.abs(d[p + 1:]).max() == 0.0 and np.abs(d[:p + 1]).max() > 0


# ------------------------------------------------------- Figure 6 golden ----
def test_figure6_prompt_workflow():
    gold = json.load(open(os.path.join(GOLDEN, "fig6_prompt_workflow.json")))
    cfg = small_cfg(tokens_per_hi_page=2, tokens_per_lo_page=4, prompt_grant_slack=0, recent_window=0,
                    n_pages=16, max_requests=1, max_seq_len=8)
    pool = oracle.Pool(cfg)
    pool.pointers[0] = gold["config"]["list_start_before"]
    # tiers chosen to give head A 2 hi + 4 lo tokens and head B 4 hi + 2 lo tokens
    tiers = {0: "HLLPHLPL", 1: "HHLHLPHP"}
    imp = {"H": 1.0, "L": 0.1, "P": 0.001}   # thresholds: 2/8 = 0.25 and 0.25/8 = 0.03125
    n0 = 8
    S = np.zeros((n0, 2), np.float32)
    for h in (0, 1):
        for j, t in enumerate(tiers[h]):
            S[j, h] = imp[t] * min(32, n0 - j)
    k = workloads.random_fp16((n0, 2, 128), 1)
    v = workloads.random_fp16((n0, 2, 128), 2)
    p_end = int(pool.pointers[1])
    assert pool.prompt(0, [0], [n0], k, v, scores_in=S) == 0
    L = pool.table_len
    for h, name in ((0, "A"), (1, "B")):
        row = pool.table[0, 0, h]
        nhi = len(gold["expected"]["hi_pages"][name]); nlo = len(gold["expected"]["lo_pages"][name])
        assert [int(x) for x in row[:nhi]] == gold["expected"]["hi_pages"][name]
        assert [int(row[L - 1 - x]) for x in range(nlo)] == gold["expected"]["lo_pages"][name]
        assert (row[nhi:L - nlo] == -1).all()
    rec = [int(pool.free_list[c % 16]) for c in range(p_end, int(pool.pointers[1]))]
    assert rec == gold["expected"]["reclaimed_in_order"]
    assert int(pool.pointers[0]) == gold["expected"]["list_start_after"]


def test_table_size_statement():
    """Bidirectional page table: 'entry length = max sequence length / tokens
    per hi page', all tables 32 MB for Llama3-8B at batch 128 (32 layers, 8 KV
    heads, int32 entries; 4096 / 16 = 256 entries). The oracle adds one entry
    so that a row can never overflow."""
    cfg = small_cfg(max_seq_len=4096, tokens_per_hi_page=16, n_layers=1, max_requests=1, n_pages=8)
    pool = oracle.Pool(cfg)
    assert pool.table_len - 1 == 256
    assert 32 * 128 * 8 * (pool.table_len - 1) * 4 == 32 * 2 ** 20


# ---------------------------------------------------- classification -------
def _prompt_with_scores(cfg, lens, S, seed=0):
    pool = oracle.Pool(cfg)
    n = int(sum(lens))
    k = workloads.random_fp16((n, cfg["n_kv_heads"], 128), seed)
    v = workloads.random_fp16((n, cfg["n_kv_heads"], 128), seed + 1)
    rc = pool.prompt(0, list(range(len(lens))), lens, k, v, scores_in=S)
    return pool, rc, k, v


def _tiers_from_pool(pool, slot, kvh, n0):
    snap = pool.snapshot()
    toks = pagefmt.head_tokens(snap, 0, slot, kvh, pool.t_hi, pool.t_lo)
    t = np.zeros(n0, np.int32)
    for r in toks["hi"]:
        t[r["pos"]] = 2
    for r in toks["lo"]:
        t[r["pos"]] = 1
    return t, toks


@pytest.mark.parametrize("case", ["all_hi", "window_only", "all_lo", "lo_disabled"])
def test_classification_special_cases(case):
    n0, W = 300, 64
    over = dict(all_hi=dict(alpha_h=0.0, alpha_l=0.0), window_only=dict(alpha_h=math.inf, alpha_l=math.inf),
                all_lo=dict(alpha_h=math.inf, alpha_l=0.0), lo_disabled=dict(lo_enabled=0, alpha_l=0.25))[case]
    cfg = small_cfg(**over)
    S = workloads.given_scores(n0, 2, seed=3, zero_frac=0.0)
    pool, rc, _, _ = _prompt_with_scores(cfg, [n0], S)
    assert rc == 0
    for h in range(2):
        t, _ = _tiers_from_pool(pool, 0, h, n0)
        win = np.arange(n0) >= n0 - W
        assert (t[win] == 2).all()
        if case == "all_hi":
            assert (t == 2).all()
        elif case == "window_only":
            assert (t[~win] == 0).all()
        elif case == "all_lo":
            assert (t[~win] == 1).all()
        else:
            assert (t != 1).all()
            imp = S[:, h] / np.minimum(32, n0 - np.arange(n0))
            keep = imp >= 0.25 / n0 * (1 + 1e-5)
            drop = imp < 0.25 / n0 * (1 - 1e-5)
            assert (t[~win & keep] == 2).all() and (t[~win & drop] == 0).all()


def test_threshold_interval_closure():
    """hi strictly above alpha_h/N; lo on the closed interval [alpha_l/N,
    alpha_h/N]; prune strictly below alpha_l/N. N = 8: thresholds 0.25 and
    0.03125 are exact in binary; count c = 8 - j."""
    cfg = small_cfg(recent_window=0, max_seq_len=8, tokens_per_hi_page=2, tokens_per_lo_page=4)
    n0 = 8
    c = np.minimum(32, n0 - np.arange(n0)).astype(np.float32)
    I = np.array([0.25, 0.25 + 2 ** -20, 0.03125, 0.03125 - 2 ** -25, 0.1, 0.0, 1.0, 0.25], np.float32)
    S = np.stack([I * c, I * c], 1).astype(np.float32)
    assert ((S[:, 0] / c) == I).all()  # chosen so that the division is exact
    pool, rc, _, _ = _prompt_with_scores(cfg, [n0], S)
    assert rc == 0
    t, _ = _tiers_from_pool(pool, 0, 0, n0)
    assert list(t) == [1, 2, 1, 0, 1, 0, 2, 1]


# ------------------------------------------------------ pages and codes ----
def test_prompt_pack_layout_and_codes():
    """Every stored token's page bytes decode to the codec's output for its
    own input vector at its tier; hi tokens in ascending position from the
    left of the grant, lo tokens from the right."""
    cfg = small_cfg(n_pages=64)
    n0 = 200
    S = workloads.given_scores(n0, 2, seed=5)
    pool, rc, k, v = _prompt_with_scores(cfg, [n0], S, seed=11)
    assert rc == 0
    for h in range(2):
        t, toks = _tiers_from_pool(pool, 0, h, n0)
        for tier, key, kb, vb in ((2, "hi", 8, 4), (1, "lo", 4, 2)):
            pos = [r["pos"] for r in toks[key]]
            assert pos == sorted(pos) and pos == list(np.nonzero(t == tier)[0])
            for r in toks[key]:
                kx = k[r["pos"], h].astype(np.float32); vx = v[r["pos"], h].astype(np.float32)
                kc, ks, kz = oracle.quantize(kx, kb)
                vc, vs, vz = oracle.quantize(vx, vb)
                assert (r["kc"] == kc).all() and (r["vc"] == vc).all()
                assert (r["ks"], r["kz"], r["vs"], r["vz"]) == (ks, kz, vs, vz)
                assert r["score"] == S[r["pos"], h]
    pagefmt.check_invariants(pool.snapshot(), pool.t_hi, pool.t_lo, cfg["n_pages"])


def test_page_format_byte_positions():
    """Spot checks of the format by absolute byte position: hi page key code
    of (slot 3, feature 5) at byte 3*128+5; value code of (slot 3, feature 6)
    in word 1 of value row 1 at bit 16 + 8; lo page key codes of features 2,3
    of slot 1 in byte 64 + 1."""
    cfg = small_cfg(recent_window=0, alpha_h=0.0, alpha_l=0.0, n_pages=8, max_seq_len=40)
    n0 = 20
    S = np.full((n0, 2), 1.0, np.float32)
    pool, rc, k, v = _prompt_with_scores(cfg, [n0], S, seed=21)
    assert rc == 0
    page = pool.pages[pool.table[0, 0, 0, 0]]
    kc, _, _ = oracle.quantize(k[3, 0].astype(np.float32), 8)
    vc, _, _ = oracle.quantize(v[3, 0].astype(np.float32), 4)
    assert page[3 * 128 + 5] == kc[5]
    vw = int(page[2304 + 128 + 4: 2304 + 128 + 8].view("<u4")[0])
    assert (vw >> (16 + 8)) & 15 == vc[6]
    cfg2 = small_cfg(recent_window=0, alpha_h=math.inf, alpha_l=0.0, n_pages=8, max_seq_len=40)
    pool2, rc, k2, v2 = _prompt_with_scores(cfg2, [n0], S, seed=21)
    L = pool2.table_len
    page2 = pool2.pages[pool2.table[0, 0, 0, L - 1]]
    kc2, _, _ = oracle.quantize(k2[1, 0].astype(np.float32), 4)
    assert page2[64 + 1] == (kc2[2] | (kc2[3] << 4))


# ----------------------------------------------------------- attention -----
def _grid_vectors(rng, n, bits, s, z):
    L = (1 << bits) - 1
    c = rng.integers(0, L + 1, size=(n, 128))
    c[:, 0], c[:, 1] = 0, L
    return (z + s * c).astype(np.float16)


def test_attention_exact_dequant_matches_dense_softmax():
    """Tokens whose K/V lie on their tier's quantization grid are stored
    losslessly, so the oracle's attention over the pages must equal dense
    fp64 softmax attention (scipy softmax, numpy matmul) over the inputs."""
    rng = np.random.default_rng(3)
    n0, H, G = 150, 2, 4
    cfg = small_cfg(recent_window=16)
    S = workloads.given_scores(n0, H, seed=9)
    # tiers depend only on the given scores: find them with a first pool, then
    # draw every token on its tier's grid for a second pool
    first, rc0, _, _ = _prompt_with_scores(cfg, [n0], S)
    assert rc0 == 0
    tiers = np.stack([_tiers_from_pool(first, 0, h, n0)[0] for h in range(H)], 1)
    pool = oracle.Pool(cfg)
    k = np.zeros((n0, H, 128), np.float16); v = np.zeros((n0, H, 128), np.float16)
    for h in range(H):
        for j in range(n0):
            hi = tiers[j, h] == 2
            k[j, h] = _grid_vectors(rng, 1, 8 if hi else 4, 2.0 ** -4, -4.0)[0]
            v[j, h] = _grid_vectors(rng, 1, 4 if hi else 2, 0.5, -2.0)[0]
    assert pool.prompt(0, [0], [n0], k, v, scores_in=S) == 0
    q = rng.standard_normal((1, H * G, 128)).astype(np.float16)
    rc, out = pool.attention(0, [0], q)
    assert rc == 0
    for h in range(H):
        keep = tiers[:, h] > 0
        K = k[keep, h].astype(np.float64); V = v[keep, h].astype(np.float64)
        for g in range(G):
            p = scipy.special.softmax(K @ q[0, h * G + g].astype(np.float64) / math.sqrt(128))
            np.testing.assert_allclose(out[0, h * G + g], p @ V, rtol=1e-12, atol=1e-12)


def test_attention_score_update_sums_to_one_for_g1():
    cfg = small_cfg(group_size=1, n_kv_heads=1)
    n0 = 100
    S = workloads.given_scores(n0, 1, seed=4)
    pool, rc, _, _ = _prompt_with_scores(cfg, [n0], S, seed=4)
    before = pool.snapshot()
    q = workloads.random_fp16((1, 1, 128), 8)
    rc, out = pool.attention(0, [0], q, update_scores=True)
    assert rc == 0
    after = pool.snapshot()
    tb = pagefmt.head_tokens(before, 0, 0, 0, pool.t_hi, pool.t_lo)
    ta = pagefmt.head_tokens(after, 0, 0, 0, pool.t_hi, pool.t_lo)
    delta = sum(a["score"] - b["score"] for key in ("hi", "lo") for a, b in zip(ta[key], tb[key]))
    assert abs(delta - 1.0) < 1e-4
    assert pool.req_state[0, 0, 3] == 1


def test_attention_uniform_logits_give_mean_value():
    cfg = small_cfg()
    n0 = 90
    S = workloads.given_scores(n0, 2, seed=6)
    pool, rc, _, _ = _prompt_with_scores(cfg, [n0], S, seed=6)
    q = np.zeros((1, 8, 128), np.float16)
    rc, out = pool.attention(0, [0], q)
    snap = pool.snapshot()
    for h in range(2):
        toks = pagefmt.head_tokens(snap, 0, 0, h, pool.t_hi, pool.t_lo)
        vs = np.stack([pagefmt.dequant(r)[1] for r in toks["hi"] + toks["lo"]])
        for g in range(4):
            np.testing.assert_allclose(out[0, h * 4 + g], vs.mean(0), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- decode -----
def _run_decode(cfg, n0, steps, S, update=True, seed=0, n_req=1):
    pool = oracle.Pool(cfg)
    H, G = cfg["n_kv_heads"], cfg["group_size"]
    lens = [n0] * n_req
    k = workloads.random_fp16((n0 * n_req, H, 128), seed)
    v = workloads.random_fp16((n0 * n_req, H, 128), seed + 1)
    assert pool.prompt(0, list(range(n_req)), lens, k, v, scores_in=S) == 0
    for t in range(steps):
        kn = workloads.random_fp16((n_req, H, 128), 100 + t)
        vn = workloads.random_fp16((n_req, H, 128), 200 + t)
        assert pool.decode(0, list(range(n_req)), kn, vn) == 0
        q = workloads.random_fp16((n_req, H * G, 128), 300 + t)
        rc, _ = pool.attention(0, list(range(n_req)), q, update_scores=update)
        assert rc == 0
        pagefmt.check_invariants(pool.snapshot(), pool.t_hi, pool.t_lo, cfg["n_pages"],
                                 reclaim=bool(cfg["reclaim_in_decode"]))
    return pool


def _positions(pool, slot, kvh):
    toks = pagefmt.head_tokens(pool.snapshot(), 0, slot, kvh, pool.t_hi, pool.t_lo)
    return sorted(r["pos"] for r in toks["hi"]), sorted(r["pos"] for r in toks["lo"])


def test_decode_only_window_survives():
    cfg = small_cfg(alpha_h=math.inf, alpha_l=math.inf, recent_window=16, max_seq_len=200)
    n0, steps = 60, 40
    pool = _run_decode(cfg, n0, steps, workloads.given_scores(n0, 2, seed=1))
    for h in range(2):
        hi, lo = _positions(pool, 0, h)
        assert hi == list(range(n0 + steps - 16, n0 + steps)) and lo == []


def test_decode_nothing_dropped_when_thresholds_zero():
    cfg = small_cfg(alpha_h=0.0, alpha_l=0.0, recent_window=8, max_seq_len=200)
    n0, steps = 50, 30
    pool = _run_decode(cfg, n0, steps, workloads.given_scores(n0, 2, seed=2, zero_frac=0.0))
    for h in range(2):
        hi, lo = _positions(pool, 0, h)
        assert hi == list(range(n0 + steps)) and lo == []


def test_decode_all_old_tokens_low_precision():
    cfg = small_cfg(alpha_h=math.inf, alpha_l=0.0, recent_window=8, max_seq_len=200)
    n0, steps = 50, 30
    pool = _run_decode(cfg, n0, steps, workloads.given_scores(n0, 2, seed=3))
    for h in range(2):
        hi, lo = _positions(pool, 0, h)
        n = n0 + steps
        assert hi == list(range(n - 8, n)) and lo == list(range(n - 8))


@pytest.mark.parametrize("reclaim", [1, 0])
def test_decode_invariants_and_free(reclaim):
    cfg = small_cfg(tokens_per_hi_page=4, tokens_per_lo_page=8, recent_window=6, n_pages=400,
                    reclaim_in_decode=reclaim, alpha_h=1.0, alpha_l=0.4, max_seq_len=200)
    n0, steps = 70, 60
    S = workloads.given_scores(n0 * 3, 2, seed=8)
    pool = _run_decode(cfg, n0, steps, S, n_req=3)
    pagefmt.check_invariants(pool.snapshot(), pool.t_hi, pool.t_lo, 400, reclaim=bool(reclaim))
    # free one request: its pages are appended hi left-to-right, then lo outer-to-inner
    tab = pool.table[0, 1].copy(); cnt = pool.head_counts[0, 1].copy()
    end0 = int(pool.pointers[1]); L = pool.table_len
    want = []
    for h in range(2):
        want += [int(x) for x in tab[h, :cnt[h, 2]]] + [int(tab[h, L - 1 - x]) for x in range(cnt[h, 3])]
    assert pool.free_request(1) == 0
    got = [int(pool.free_list[c % 400]) for c in range(end0, int(pool.pointers[1]))]
    assert got == want
    assert pool.free_request(1) == oracle.ERR["STATE"]
    for s in (0, 2):
        assert pool.free_request(s) == 0
    snap = pool.snapshot()
    assert int(snap["pointers"][1] - snap["pointers"][0]) == 400 and (snap["table"] == -1).all()


def test_errors_are_no_ops():
    cfg = small_cfg(n_pages=20)
    pool = oracle.Pool(cfg)
    n0 = 400                                 # needs 2 heads x (23 + 1) pages > 20
    before = pool.snapshot()
    S = workloads.given_scores(n0, 2, seed=1)
    k = workloads.random_fp16((n0, 2, 128), 1); v = workloads.random_fp16((n0, 2, 128), 2)
    assert pool.prompt(0, [0], [n0], k, v, scores_in=S) == oracle.ERR["NO_PAGES"]
    after = pool.snapshot()
    for key in before:
        assert (before[key] == after[key]).all()
    assert pool.prompt(0, [0], [0], k, v, scores_in=S) == oracle.ERR["ARG"]
    assert pool.decode(0, [0], k[:1], v[:1]) == oracle.ERR["STATE"]
    # slack 0 can leave a head one page short: detected before any write
    cfg2 = small_cfg(tokens_per_hi_page=2, tokens_per_lo_page=4, prompt_grant_slack=0, recent_window=0,
                     max_seq_len=8)
    pool2 = oracle.Pool(cfg2)
    S2 = np.zeros((2, 2), np.float32); S2[0] = 10.0; S2[1] = 0.2   # one hi token, one lo token
    k2 = workloads.random_fp16((2, 2, 128), 3)
    before = pool2.snapshot()
    assert pool2.prompt(0, [0], [2], k2, k2, scores_in=S2) == oracle.ERR["TABLE_FULL"]
    after = pool2.snapshot()
    for key in before:
        assert (before[key] == after[key]).all()


# ------------------------------------------------- per-head thresholds -----
def _head_records(pool, slot, kvh):
    """A head's stored tokens, tier by tier in slot order, without page IDs."""
    toks = pagefmt.head_tokens(pool.snapshot(), 0, slot, kvh, pool.t_hi, pool.t_lo)
    key = lambda r: (r["pos"], tuple(r["kc"]), tuple(r["vc"]), r["ks"], r["kz"], r["vs"], r["vz"],
                     np.float32(r["score"]).view(np.uint32).item())
    return [key(r) for r in toks["hi"]], [key(r) for r in toks["lo"]]


def test_per_head_thresholds_equal_uniform_pools_head_by_head():
    """Compaction policy, extensibility (thresholds for each head on its
    own): a pool whose two KV heads carry different (alpha_h, alpha_l) stores,
    head by head, exactly what a pool configured with that head's pair for
    every head stores, through a prompt and generation steps with score
    updates (the attention of a KV head sees only its own tokens)."""
    pairs = [(2.0, 0.25), (0.8, 0.5)]
    base = small_cfg(recent_window=8, max_seq_len=400, n_pages=512, tokens_per_hi_page=4, tokens_per_lo_page=8)
    n0, steps, H, G = 150, 25, 2, 4
    k = workloads.random_fp16((n0, H, 128), 31)
    v = workloads.random_fp16((n0, H, 128), 32)
    S = workloads.given_scores(n0, H, seed=33, scale=0.5)
    pools = [oracle.Pool(base)] + [oracle.Pool(dict(base, alpha_h=a, alpha_l=b)) for a, b in pairs]
    assert pools[0].set_thresholds(0, [a for a, _ in pairs], [b for _, b in pairs]) == 0
    assert (pools[0].thresholds[0] == np.array(pairs, np.float32)).all()
    for p in pools:
        assert p.prompt(0, [0], [n0], k, v, scores_in=S) == 0
    for t in range(steps):
        kn = workloads.random_fp16((1, H, 128), 400 + t)
        vn = workloads.random_fp16((1, H, 128), 500 + t)
        q = workloads.random_fp16((1, H * G, 128), 600 + t)
        for p in pools:
            assert p.decode(0, [0], kn, vn) == 0
            assert p.attention(0, [0], q, update_scores=True)[0] == 0
        for h in range(H):
            assert _head_records(pools[0], 0, h) == _head_records(pools[1 + h], 0, h), (t, h)
    # the two pairs really differ in what they keep
    assert _head_records(pools[1], 0, 0) != _head_records(pools[2], 0, 0)
    assert pools[0].set_thresholds(0, [np.nan, 1.0], [0.1, 0.1]) == oracle.ERR["ARG"]
    assert pools[0].set_thresholds(1, [1.0, 1.0], [0.1, 0.1]) == oracle.ERR["ARG"]


# ------------------------------------------------------ prefill attention ---
def _dense_causal(q, k, v):
    """numpy / scipy causal attention: q [N, G, 128], k, v [N, 128] (float64)."""
    n, G = q.shape[0], q.shape[1]
    logits = np.einsum("pgf,jf->pgj", q, k) / np.sqrt(128.0)
    mask = np.tril(np.ones((n, n), bool))[:, None, :]
    logits = np.where(mask, logits, -np.inf)
    p = scipy.special.softmax(logits, axis=-1)
    lse = scipy.special.logsumexp(logits, axis=-1)
    return np.einsum("pgj,jf->pgf", p, v), lse / np.log(2.0)


@pytest.mark.parametrize("n0,G", [(1, 1), (37, 3), (130, 4)])
def test_prefill_attention_matches_scipy(n0, G):
    q = workloads.random_fp16((n0, G, 128), 700 + n0, scale=1.5)
    k = workloads.random_fp16((n0, 128), 701 + n0)
    v = workloads.random_fp16((n0, 128), 702 + n0)
    out, lse2 = oracle.prefill_attention(q, k, v)
    ref, rlse = _dense_causal(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64))
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse2, rlse, rtol=1e-12, atol=1e-12)


def test_prefill_attention_equal_keys_and_causality():
    """Equal keys: every visible key has the same weight, so row p's output is
    the mean of v[0..p] and its base-2 log-sum-exp is log2(p + 1) + q.k /
    (sqrt(128) ln 2); changing later values changes no earlier row."""
    n0, G = 50, 2
    q = workloads.random_fp16((n0, G, 128), 710)
    krow = workloads.random_fp16((1, 128), 711)
    k = np.repeat(krow, n0, axis=0)
    v = workloads.random_fp16((n0, 128), 712)
    out, lse2 = oracle.prefill_attention(q, k, v)
    vd = v.astype(np.float64)
    means = np.cumsum(vd, axis=0) / np.arange(1, n0 + 1)[:, None]
    for g in range(G):
        np.testing.assert_allclose(out[:, g], means, rtol=1e-12, atol=1e-12)
        qk = q[:, g].astype(np.float64) @ krow[0].astype(np.float64) / np.sqrt(128.0)
        np.testing.assert_allclose(lse2[:, g], np.log2(np.arange(1, n0 + 1)) + qk / np.log(2.0), rtol=1e-12,
                                   atol=1e-12)
    v2 = v.copy()
    v2[30:] = workloads.random_fp16((n0 - 30, 128), 713)
    out2, _ = oracle.prefill_attention(q, k, v2)
    assert (out2[:30] == out[:30]).all() and not (out2[30:] == out[30:]).all()


def test_prefill_rows_match_scipy_and_the_full_prompt():
    """Selected rows: each equals the scipy row at its position (keys 0..p),
    and the same row of the whole-prompt computation bit for bit."""
    n0, G = 90, 3
    q = workloads.random_fp16((n0, G, 128), 720, scale=1.5)
    k = workloads.random_fp16((n0, 128), 721)
    v = workloads.random_fp16((n0, 128), 722)
    pos = np.array([0, 89, 17, 45, 45, 63])
    out, lse2 = oracle.prefill_rows(pos, q[pos], k, v)
    ref, rlse = _dense_causal(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64))
    np.testing.assert_allclose(out, ref[pos], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse2, rlse[pos], rtol=1e-12, atol=1e-12)
    full, flse = oracle.prefill_attention(q, k, v)
    assert (out == full[pos]).all() and (lse2 == flse[pos]).all()
    # keys after the largest position are never read
    k2, v2 = k.copy(), v.copy()
    k2[64:], v2[64:] = 1000.0, -1000.0
    out3, _ = oracle.prefill_rows(pos[pos < 64], q[pos[pos < 64]], k2, v2)
    assert (out3 == out[pos < 64]).all()

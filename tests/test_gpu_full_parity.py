"""GPU parity at the workloads' full sizes, element by element.

- Prompt with caller scores, every head of the llama8b batch (256 heads), of a
  batch of 800 heads in shuffled slot order (the grant and reclaim prefix sums
  over more heads than one thread block holds, several heads a thread) and of
  the Qwen2.5-7B-shaped batch (128 requests x U{1K..16K}, 512 heads, low tier
  off): the whole exported state is bit-exact against the oracle
  (free list, pointers, table, counters, request state, every valid page bit).
- Prompt with scores computed from the observation queries on the llama8b and
  llama70b batches, where each persistent tensor-core CTA scores dozens of
  128-key tiles across several heads: every score within the score tolerance
  of the oracle's fp64 scores; the oracle fed the GPU's own fp32 scores
  reproduces the GPU state bit for bit; tiers agree with the fp64 scores'
  tiers outside the tie band that the score tolerance implies.
- The generation loop the benchmark times (compaction, then attention with
  the score update, every step): before a step the oracle takes over the GPU's
  state, both run the step, and the states must be identical; attention
  outputs and updated scores are compared with the oracle's fp64 attention
  over the same state. Heads hold more than 4096 tokens, so the victim search
  runs on several CTAs per head.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import workloads
from tests import parity
from tests.gpu_pool import GPool, load_into, stored

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ATT_ATOL, ATT_RTOL = 1e-3, 2e-3       # attention output vs fp64
SC_ATOL, SC_RTOL = 1e-6, 5e-5         # prompt scores vs fp64 (fp32 tensor-core logits, exp2)
UPD_ATOL, UPD_RTOL = 1e-6, 1e-4       # updated scores: one fp32 add of a probability
# Tie band, from the score tolerance: a GPU score within SC_ATOL + SC_RTOL*S of
# the fp64 score gives an importance within that error over c (plus the fp32
# roundings of I and of alpha/N, 2^-22 relative), so only tokens whose fp64
# importance lies that close to a threshold may land on the other side.
ROUND_REL = 2.0 ** -22


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiated_kv_cache_gb300 as dkv
    dkv.build.build()
    dkv.load()


def _compare(gp, op, **kw):
    parity.compare_states(gp.snapshot(), op.snapshot(), gp.t_hi, gp.t_lo, gp.cfg["n_pages"],
                          gp.cfg["page_bytes"], table_len=gp.table_len, t_mid=gp.t_mid, **kw)


# -------------------------------------------------- prompt, caller scores
def _many_heads_batch():
    rng = np.random.default_rng(2024)
    R, H = 100, 8
    lens = rng.integers(40, 1201, size=R).astype(np.int32)
    n = int(lens.sum())
    k = workloads.random_fp16((n, H, 128), 71, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 72)
    cfg = dict(n_layers=1, n_kv_heads=H, group_size=4, head_dim=128, page_bytes=3584, n_pages=60000,
               max_requests=R + 7, max_seq_len=1300, tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=1,
               alpha_h=2.0, alpha_l=0.25, recent_window=64, obs_window=32, prompt_grant_slack=1,
               reclaim_in_decode=1)
    slots = rng.permutation(R + 7)[:R].astype(np.int32)
    return cfg, [int(s) for s in slots], [int(x) for x in lens], k, v


@pytest.mark.parametrize("name", ["llama8b", "many_heads", "qwen7b"])
def test_prompt_given_scores_full_size(name):
    if name == "many_heads":
        cfg, slots, lens, k, v = _many_heads_batch()
    else:
        w = workloads.WORKLOADS[name]
        inp = workloads.prompt_inputs(name, 0)
        cfg = w.pool_config()
        lens = [int(x) for x in inp["lens"]]
        slots = list(range(w.n_requests))
        k, v = inp["k"], inp["v"]
    H = cfg["n_kv_heads"]
    S = workloads.given_scores(sum(lens), H, seed=11, scale=0.02)
    print(f"{name}: {len(lens)} requests x {H} KV heads = {len(lens) * H} heads, {sum(lens)} tokens")
    with GPool(cfg) as gp:
        rc, so = gp.prompt(0, slots, lens, k, v, scores_in=S, want_scores=True)
        assert (so == S).all()
        st = gp.status()
        assert st["error"] == 0, st
        op = oracle.Pool(cfg)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        _compare(gp, op)
        print(f"{name}: hi {st['hi_tokens']} lo {st['lo_tokens']} tokens, {st['free_pages']} pages free")


# ------------------------------------------------ prompt, computed scores
def _fp64_scores(inp, H, G, lens, workers=16):
    jobs, t0 = [], 0
    for i, n0 in enumerate(lens):
        for h in range(H):
            jobs.append((t0, n0, i, h))
        t0 += n0
    S64 = np.zeros((t0, H))

    def one(job):
        t, n0, i, h = job
        S64[t:t + n0, h] = oracle.unit_scores(inp["k"][t:t + n0, h], inp["q_obs"][i][:, h * G:(h + 1) * G])

    with ThreadPoolExecutor(max_workers=workers) as ex:      # the oracle's C code runs without the GIL
        list(ex.map(one, jobs))
    return S64


def _tie_band(S64, lens, H, cfg):
    ties = np.zeros(S64.shape, bool)
    alphas = [cfg["alpha_h"], cfg["alpha_l"]] if cfg["lo_enabled"] else [cfg["alpha_l"]]
    t0 = 0
    for n0 in lens:
        j = np.arange(n0)
        c = np.minimum(32, n0 - j)[:, None].astype(np.float64)
        IN = S64[t0:t0 + n0] / c * n0                       # importance x N, against alpha
        err = (SC_RTOL + ROUND_REL) * IN + SC_ATOL / c * n0
        near = np.zeros_like(IN, bool)
        for a in alphas:
            if np.isfinite(a) and a > 0:
                near |= np.abs(IN - a) <= err + ROUND_REL * a
        near[j >= n0 - cfg["recent_window"]] = False
        ties[t0:t0 + n0] = near
        t0 += n0
    return ties


@pytest.mark.parametrize("name", ["llama8b", "llama70b"])
def test_prompt_computed_scores_full_size(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.prompt_inputs(name, 0)
    cfg = w.pool_config()
    H, G = w.n_kv_heads, w.group_size
    lens = [int(x) for x in inp["lens"]]
    slots = list(range(w.n_requests))
    tiles = sum(-(-n0 // 128) for n0 in lens) * H
    print(f"{name}: {tiles} key tiles over the persistent tensor-core grid")
    with GPool(cfg) as gp:
        rc, so = gp.prompt(0, slots, lens, inp["k"], inp["v"], inp["q_obs"], want_scores=True)
        assert gp.status()["error"] == 0
        gsnap = gp.snapshot()
    S64 = _fp64_scores(inp, H, G, lens)
    ok, worst = parity.within(so.astype(np.float64), S64, SC_ATOL, SC_RTOL)
    rel = np.abs(so - S64) / np.maximum(S64, 1e-30)
    print(f"{name}: score max rel err {rel.max():.3e}, tolerance excess {worst:.3e}")
    assert ok, worst
    # (i) the oracle fed the GPU's own scores reproduces the GPU state bit for bit
    op = oracle.Pool(cfg)
    assert op.prompt(0, slots, lens, inp["k"], inp["v"], scores_in=so) == 0
    parity.compare_states(gsnap, op.snapshot(), gp.t_hi, gp.t_lo, cfg["n_pages"], cfg["page_bytes"])
    del op
    # (iii) tiers against the fp64 scores' tiers, outside the tie band
    ties = _tie_band(S64, lens, H, cfg)
    op64 = oracle.Pool(cfg)
    assert op64.prompt(0, slots, lens, inp["k"], inp["v"], scores_in=S64.astype(np.float32)) == 0
    osnap = op64.snapshot()
    t0 = 0
    for i, n0 in enumerate(lens):
        for h in range(H):
            tg = _tiers(gsnap, (0, i, h), n0, gp.t_hi, gp.t_lo)
            to = _tiers(osnap, (0, i, h), n0, gp.t_hi, gp.t_lo)
            tie = ties[t0:t0 + n0, h]
            assert (tg[~tie] == to[~tie]).all(), f"tier differs outside the tie band (req {i}, head {h})"
        t0 += n0
    print(f"{name}: {int(ties.sum())} of {ties.size} token-heads in the tie band")


def _tiers(snap, head, n, t_hi, t_lo):
    hi, lo = stored(snap, head, t_hi, t_lo, 5, np.int32)
    t = np.zeros(n, np.int8)
    t[hi] = 2
    t[lo] = 1
    return t


# ------------------------------------------------------- generation loop
def _step_and_compare(gp, op, slots, kn, vn):
    """One generation-phase step on both sides from the GPU's current state."""
    load_into(op, gp.snapshot())
    gp.decode(0, slots, kn, vn)
    assert op.decode(0, slots, kn, vn) == 0
    assert gp.status()["error"] == 0
    _compare(gp, op)


def _attention_and_compare(gp, op, slots, q, G):
    """Attention with the score update on both sides from the GPU's state:
    outputs within the attention tolerance of fp64, updated scores within
    one fp32 rounding of the fp64 update, update counters identical."""
    before = gp.snapshot()
    load_into(op, before)
    out = gp.attention(0, slots, q, update=True)
    rc, ref = op.attention(0, slots, q, update_scores=True)
    assert rc == 0
    ok, worst = parity.within(out.astype(np.float64), ref, ATT_ATOL, ATT_RTOL)
    assert ok, worst
    after, osnap = gp.snapshot(), op.snapshot()
    assert (after["req_state"] == osnap["req_state"]).all()
    H = gp.cfg["n_kv_heads"]
    for i, s in enumerate(slots):
        for h in range(H):
            for a, b in zip(stored(after, (0, s, h), gp.t_hi, gp.t_lo, 4, np.float32),
                            stored(osnap, (0, s, h), gp.t_hi, gp.t_lo, 4, np.float32)):
                ok, worst = parity.within(a.astype(np.float64), b.astype(np.float64), UPD_ATOL, UPD_RTOL)
                assert ok, (s, h, worst)
    return float((np.abs(out - ref) / (ATT_ATOL + ATT_RTOL * np.abs(ref))).max())


@pytest.mark.parametrize("G,pb", [(4, 3584), (8, 4096)])
def test_generation_loop_with_score_updates(G, pb):
    """96 steps of (compaction, attention with score update) on heads of up
    to 9000 tokens, compared with the oracle at every step."""
    H, lens, slots = 2, [9000, 5000, 700], [2, 0, 1]
    cfg = dict(n_layers=1, n_kv_heads=H, group_size=G, head_dim=128, page_bytes=pb, n_pages=8000,
               max_requests=3, max_seq_len=9200, tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=1,
               alpha_h=2.0, alpha_l=0.25, recent_window=64, obs_window=32, prompt_grant_slack=1,
               reclaim_in_decode=1)
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 81, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 82)
    # prompt scores spread around the thresholds, so decode keeps demoting and
    # pruning; the longest heads keep more than 2 x 2048 tokens (three scan CTAs)
    S = workloads.given_scores(n, H, seed=83, scale=0.2)
    op = oracle.Pool(cfg)
    worst = 0.0
    with GPool(cfg) as gp:
        gp.prompt(0, slots, lens, k, v, scores_in=S)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        _compare(gp, op)
        stored_max = int(gp.snapshot(pages=False)["head_counts"][..., :2].sum(-1).max())
        assert stored_max > 2 * 2048, stored_max
        moved = 0
        for step in range(96):
            kn = workloads.random_fp16((3, H, 128), 900 + step)
            vn = workloads.random_fp16((3, H, 128), 1900 + step)
            q = workloads.random_fp16((3, H * G, 128), 2900 + step, scale=2.0)
            c0 = gp.snapshot(pages=False)["head_counts"].copy()
            _step_and_compare(gp, op, slots, kn, vn)
            moved += int((gp.snapshot(pages=False)["head_counts"][..., 1] != c0[..., 1]).sum())
            worst = max(worst, _attention_and_compare(gp, op, slots, q, G))
        st = gp.status()
        assert st["error"] == 0
        print(f"G={G}: 96 steps bit-exact (longest head {stored_max} tokens); {moved} head-steps changed the lo tier; "
              f"attention max err/tolerance {worst:.3f}; stored hi {st['hi_tokens']} lo {st['lo_tokens']}")
        assert moved > 0
        for s in slots:
            gp.free(s)
            assert op.free_request(s) == 0
        _compare(gp, op)


@pytest.mark.parametrize("three", [False, True])
def test_benchmark_loop_llama8b(three):
    """The benchmark's own step on the full llama8b batch: prompt with
    computed scores, then 128 x (compaction, attention with score update).
    At sampled steps the oracle takes over the GPU's state and both run the
    compaction; the states must be identical. Also with the three-tier pool
    the benchmark runs as `llama8b+mid` (mid tier K8V2 from 1/N)."""
    name = "llama8b"
    w = workloads.WORKLOADS[name]
    inp = workloads.prompt_inputs(name, 0)
    cfg = w.pool_config(**(workloads.THREE_TIER if three else {}))
    R, H = w.n_requests, w.n_kv_heads
    slots = list(range(R))
    lens = [int(x) for x in inp["lens"]]
    check = {0, 1, 2, 3, 31, 64, 100, 127}
    op = oracle.Pool(cfg)
    with GPool(cfg) as gp:
        gp.prompt(0, slots, lens, inp["k"], inp["v"], inp["q_obs"])
        for t in range(w.decode_steps):
            d = workloads.decode_inputs(name, t)
            if t in check:
                _step_and_compare(gp, op, slots, d["k"], d["v"])
            else:
                gp.decode(0, slots, d["k"], d["v"])
            gp.attention(0, slots, d["q"], update=True)
        st = gp.status()
        assert st["error"] == 0
        assert int(gp.snapshot(pages=False)["req_state"][0, 0, 3]) == w.decode_steps
        print(f"llama8b{'+mid' if three else ''}: {len(check)} steps compared; stored hi {st['hi_tokens']} "
              f"mid {st['mid_tokens']} lo {st['lo_tokens']}")
        if three:
            assert st["mid_tokens"] > 0


def test_generation_steps_after_mixed_attention_calls():
    """Generation steps whose previous attention calls vary: score updates on
    every request, on a subset, twice in a row, followed by a call without
    update, through the allocation-free entry point, or no attention at all.
    A step takes the victim keys a call's score update left only while the
    request is as that call left it, and otherwise searches the head; every
    step is compared with the oracle from the GPU's state."""
    import differentiated_kv_cache_gb300 as dkv
    H, G, lens, slots = 2, 4, [3000, 500, 40], [0, 1, 2]
    cfg = dict(n_layers=2, n_kv_heads=H, group_size=G, head_dim=128, page_bytes=3584, n_pages=3000,
               max_requests=3, max_seq_len=3200, tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=1,
               alpha_h=2.0, alpha_l=0.25, recent_window=16, obs_window=32, prompt_grant_slack=1,
               reclaim_in_decode=1)
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 91, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 92)
    S = workloads.given_scores(n, H, seed=93, scale=0.2)
    op = oracle.Pool(cfg)

    def attend(gp, layer, sl, step, update, static=False):
        q = gp.dev(workloads.random_fp16((len(sl), H * G, 128), 3000 + 10 * step + len(sl), scale=2.0))
        out = torch.empty((len(sl), H * G, 128), dtype=torch.float32, device="cuda")
        f = dkv.dkv_decode_attention_static if static else dkv.dkv_decode_attention
        f(gp.h, layer, sl, q, out, update)
        torch.cuda.synchronize()

    with GPool(cfg) as gp:
        for layer in (0, 1):
            gp.prompt(layer, slots, lens, k, v, scores_in=S)
        for step in range(40):
            layer = step % 2
            kn = workloads.random_fp16((3, H, 128), 4000 + step)
            vn = workloads.random_fp16((3, H, 128), 5000 + step)
            load_into(op, gp.snapshot())
            gp.decode(layer, slots, kn, vn)
            assert op.decode(layer, slots, kn, vn) == 0
            assert gp.status()["error"] == 0
            _compare(gp, op)
            kind = (step // 2) % 6
            if kind == 0:
                attend(gp, layer, slots, step, True)
            elif kind == 1:
                attend(gp, layer, [2, 0], step, True)
                attend(gp, layer, slots, step, False)
            elif kind == 2:
                attend(gp, layer, slots, step, True)
                attend(gp, layer, [1], step, True)
            elif kind == 3:
                attend(gp, layer, slots, step, True, static=True)
            elif kind == 4:
                attend(gp, layer, [1, 2], step, True)
                attend(gp, 1 - layer, slots, step, True)
            # kind 5: no attention before the next step of this layer
        print("40 generation steps bit-exact after mixed attention calls")

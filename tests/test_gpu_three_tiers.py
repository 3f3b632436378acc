"""GPU parity of the three-tier pool (DiffKV, Compaction policy:
extensibility to more precision levels; Memory management, generation
workflow: further levels by combining one-way and two-way page tables).

The mid tier K8V2 sits between hi K8V4 and lo K4V2; its pages live in a
one-way table after each head's two-way one. Every kernel of the path runs
with it: classification and the prompt's prefix sums and pack, the
generation step with its demotion chain (hi -> mid, hi -> lo, mid -> lo),
the paged attention kernel's third page type, the epilogue's score update
and victim keys, and request completion. Everything integer is compared bit
for bit with the oracle; attention within 1e-3 + 2e-3 |ref| of the oracle's
fp64 attention over the same pages, updated scores within 1e-6 + 1e-4 rel.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tests import pagefmt, parity
from tests.gpu_pool import GPool, load_into

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ATT_ATOL, ATT_RTOL = 1e-3, 2e-3
UPD_ATOL, UPD_RTOL = 1e-6, 1e-4
SC_ATOL, SC_RTOL = 1e-6, 5e-5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiated_kv_cache_gb300 as dkv
    dkv.build.build()
    dkv.load()


def cfg3(**kw):
    c = dict(n_layers=1, n_kv_heads=2, group_size=4, head_dim=128, page_bytes=3584, n_pages=6000,
             max_requests=4, max_seq_len=5300, tokens_per_hi_page=0, tokens_per_lo_page=0, tokens_per_mid_page=16,
             lo_enabled=1, mid_enabled=1, alpha_h=2.0, alpha_m=0.8, alpha_l=0.25, recent_window=64, obs_window=32,
             prompt_grant_slack=2, reclaim_in_decode=1)
    c.update(kw)
    return c


def geo(gp):
    return dict(t_hi=gp.t_hi, t_lo=gp.t_lo, t_mid=gp.t_mid, table_len=gp.table_len)


def compare(gp, op, **kw):
    parity.compare_states(gp.snapshot(), op.snapshot(), gp.t_hi, gp.t_lo, gp.cfg["n_pages"], gp.cfg["page_bytes"],
                          table_len=gp.table_len, t_mid=gp.t_mid, **kw)


def test_three_tier_configuration_checks():
    import differentiated_kv_cache_gb300 as dkv
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_pool_create(dkv.make_config(**cfg3(lo_enabled=0)), 0)
    assert e.value.code == dkv.DKV_ERR_ARG
    # 4 KB pages hold 18 hi tokens: not whole 16-token chunks
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_pool_create(dkv.make_config(**cfg3(page_bytes=4096)), 0)
    assert e.value.code == dkv.DKV_ERR_UNSUPPORTED
    # the largest mid page at 3.5 KB holds 20 tokens
    with pytest.raises(dkv.DkvError) as e:
        dkv.dkv_pool_create(dkv.make_config(**cfg3(tokens_per_mid_page=0)), 0)
    assert e.value.code == dkv.DKV_ERR_UNSUPPORTED
    with GPool(cfg3(mid_enabled=0)) as gp:
        assert gp.geom["t_mid"] == 0 and gp.row_len == gp.table_len and gp.cstride == 4
        assert dkv.dkv_pool_set_mid_thresholds(gp.h, 0, [1.0, 1.0], check=False) == dkv.DKV_ERR_ARG
    with GPool(cfg3()) as gp:
        op = oracle.Pool(cfg3())
        assert (gp.t_hi, gp.t_lo, gp.t_mid) == (op.t_hi, op.t_lo, op.t_mid) == (16, 32, 16)
        assert gp.geom["mid_off"] == list(op.mid_off) and gp.geom["mid_used"] == op.mid_used
        assert gp.row_len == op.row_len and gp.geom["mid_table_len"] == op.mid_len and gp.cstride == 8


def _batch(seed, lens, H, scale=0.35):
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 10 * seed + 1, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 10 * seed + 2)
    S = workloads.given_scores(n, H, seed=10 * seed + 3, scale=scale)
    return k, v, S


@pytest.mark.parametrize("G", [4, 8, 5])
def test_prompt_given_scores_three_tiers(G):
    """Prompt with caller scores, per-head thresholds on all three levels:
    the whole exported state (list, pointers, both table parts, counters,
    every valid page bit of hi, mid and lo pages) is bit-exact."""
    H, lens, slots = 3, [3000, 517, 33, 1290], [2, 0, 3, 1]
    cfg = cfg3(n_kv_heads=H, group_size=G)
    k, v, S = _batch(G, lens, H)
    op = oracle.Pool(cfg)
    ah, am, al = [2.0, 1.5, 3.0], [0.8, 1.0, 1.2], [0.25, 0.4, 0.1]
    with GPool(cfg) as gp:
        import differentiated_kv_cache_gb300 as dkv
        dkv.dkv_pool_set_thresholds(gp.h, 0, ah, al)
        dkv.dkv_pool_set_mid_thresholds(gp.h, 0, am)
        assert op.set_thresholds(0, ah, al) == 0 and op.set_mid_thresholds(0, am) == 0
        gp.prompt(0, slots, lens, k, v, scores_in=S)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        compare(gp, op)
        st = gp.status()
        assert st["error"] == 0 and st["hi_tokens"] > 0 and st["mid_tokens"] > 0 and st["lo_tokens"] > 0, st
        snap = gp.snapshot(pages=False)
        pagefmt.check_invariants(snap, gp.t_hi, gp.t_lo, cfg["n_pages"], table_len=gp.table_len, t_mid=gp.t_mid)
        print(f"G={G}: hi {st['hi_tokens']} mid {st['mid_tokens']} lo {st['lo_tokens']} pages "
              f"{st['hi_pages']}/{st['mid_pages']}/{st['lo_pages']}")


def test_prompt_computed_scores_three_tiers():
    """Prompt scored from the observation queries on the tensor cores: scores
    within the score tolerance of the oracle's fp64 scores, and the oracle
    fed the GPU's fp32 scores reproduces the three-tier state bit for bit."""
    H, G, lens, slots = 2, 4, [2100, 700, 45], [0, 1, 2]
    cfg = cfg3(n_kv_heads=H, group_size=G)
    n = sum(lens)
    k = workloads.random_fp16((n, H, 128), 51, scale=1.5)
    v = workloads.random_fp16((n, H, 128), 52)
    q_obs = workloads.random_fp16((len(lens), 32, H * G, 128), 53, scale=2.0)
    with GPool(cfg) as gp:
        rc, so = gp.prompt(0, slots, lens, k, v, q_obs=q_obs, want_scores=True)
        t0 = 0
        for i, n0 in enumerate(lens):
            for h in range(H):
                S64 = oracle.unit_scores(k[t0:t0 + n0, h], q_obs[i][:, h * G:(h + 1) * G])
                ok, worst = parity.within(so[t0:t0 + n0, h].astype(np.float64), S64, SC_ATOL, SC_RTOL)
                assert ok, (i, h, worst)
            t0 += n0
        op = oracle.Pool(cfg)
        assert op.prompt(0, slots, lens, k, v, scores_in=so) == 0
        compare(gp, op)
        assert gp.status()["mid_tokens"] > 0


def _attention_and_compare(gp, op, slots, q, update=True, static=False):
    import differentiated_kv_cache_gb300 as dkv
    before = gp.snapshot()
    load_into(op, before)
    if static:
        qd = gp.dev(q)
        out_t = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        dkv.dkv_decode_attention_static(gp.h, 0, slots, qd, out_t, update)
        torch.cuda.synchronize()
        out = out_t.cpu().numpy()
    else:
        out = gp.attention(0, slots, q, update=update)
    rc, ref = op.attention(0, slots, q, update_scores=update)
    assert rc == 0
    ok, worst = parity.within(out.astype(np.float64), ref, ATT_ATOL, ATT_RTOL)
    assert ok, worst
    after, osnap = gp.snapshot(), op.snapshot()
    assert (after["req_state"] == osnap["req_state"]).all()
    for s in slots:
        for h in range(gp.cfg["n_kv_heads"]):
            a = pagefmt.tier_values(after, (0, s, h), geo(gp), 4, np.float32)
            b = pagefmt.tier_values(osnap, (0, s, h), geo(gp), 4, np.float32)
            for tier in a:
                ok, worst = parity.within(a[tier].astype(np.float64), b[tier].astype(np.float64), UPD_ATOL,
                                          UPD_RTOL)
                assert ok, (s, h, tier, worst)
    return float((np.abs(out - ref) / (ATT_ATOL + ATT_RTOL * np.abs(ref))).max())


@pytest.mark.parametrize("G", [4, 8, 7])
def test_generation_loop_three_tiers(G):
    """80 steps of (compaction, attention with score update) with the mid
    tier, every step compared with the oracle from the GPU's state; the
    longest head keeps more than 2 x 2048 tokens (three scan CTAs when the
    victim keys are not cached). Counts of hi -> mid, mid -> lo and hi -> lo
    movements are reported; each must occur."""
    H, lens, slots = 2, [8000, 1200, 300], [2, 0, 1]
    cfg = cfg3(n_kv_heads=H, group_size=G, max_requests=3, max_seq_len=8200)
    k, v, S = _batch(G + 20, lens, H, scale=0.3)
    op = oracle.Pool(cfg)
    worst, grew = 0.0, {"mid": 0, "lo": 0}
    with GPool(cfg) as gp:
        gp.prompt(0, slots, lens, k, v, scores_in=S)
        assert op.prompt(0, slots, lens, k, v, scores_in=S) == 0
        compare(gp, op)
        cmax = gp.snapshot(pages=False)["head_counts"]
        assert int((cmax[..., 0] + cmax[..., 1] + cmax[..., 4]).max()) > 2 * 2048
        for step in range(80):
            kn = workloads.random_fp16((3, H, 128), 900 + step)
            vn = workloads.random_fp16((3, H, 128), 1900 + step)
            q = workloads.random_fp16((3, H * G, 128), 2900 + step, scale=2.0)
            c0 = gp.snapshot(pages=False)["head_counts"].copy()
            load_into(op, gp.snapshot())
            gp.decode(0, slots, kn, vn)
            assert op.decode(0, slots, kn, vn) == 0
            assert gp.status()["error"] == 0
            compare(gp, op)
            c1 = gp.snapshot(pages=False)["head_counts"]
            grew["mid"] += int((c1[..., 4] > c0[..., 4]).sum())
            grew["lo"] += int((c1[..., 1] > c0[..., 1]).sum())
            worst = max(worst, _attention_and_compare(gp, op, slots, q, update=True, static=(step % 10 == 9)))
        st = gp.status()
        assert st["error"] == 0
        print(f"G={G}: 80 steps bit-exact; head-steps that grew mid {grew['mid']}, lo {grew['lo']}; "
              f"attention max err/tolerance {worst:.3f}; hi {st['hi_tokens']} mid {st['mid_tokens']} "
              f"lo {st['lo_tokens']}")
        assert grew["mid"] > 0 and grew["lo"] > 0
        # attention without score update, then request completion
        q = workloads.random_fp16((3, H * G, 128), 7777, scale=2.0)
        _attention_and_compare(gp, op, slots, q, update=False)
        for s in [1, 2, 0]:
            load_into(op, gp.snapshot())
            gp.free(s)
            assert op.free_request(s) == 0
            compare(gp, op)
        pagefmt.check_invariants(gp.snapshot(pages=False), gp.t_hi, gp.t_lo, cfg["n_pages"],
                                 table_len=gp.table_len, t_mid=gp.t_mid)

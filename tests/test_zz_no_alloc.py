"""dkv_decode_attention_static, the allocation-free decode attention, against
dkv_decode_attention through the C ABI, and against the oracle.

The static variant works in one fixed device array shared by every call, so
the checks run two calls in a row (the second sees the first's leftovers)
and compare each against the pool-scratch entry point on a twin pool holding
the same state; the device's free memory must not change across any static
call. This file is collected last so that, in a full run, the array has also
seen every earlier use in the process."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tests.gpu_pool import GPool, load_into, stored
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATT_ATOL, ATT_RTOL = 1e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def cfg_of(**over):
    c = dict(n_layers=1, n_kv_heads=2, group_size=4, head_dim=128, page_bytes=4096, n_pages=2048,
             max_requests=3, max_seq_len=1200, tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=1,
             alpha_h=2.0, alpha_l=0.25, recent_window=64, obs_window=32, prompt_grant_slack=1,
             reclaim_in_decode=1)
    c.update(over)
    return c


FREE_SEEN = []     # device free bytes around every static call: (before, after)


def attend(gp, fn, slots, q, update):
    """One attention call; around a static call the device's free memory is
    recorded with everything the call uses already allocated."""
    import differentiated_kv_cache_gb300 as dkv
    qd = gp.dev(q)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    before = torch.cuda.mem_get_info()[0]
    rc = getattr(dkv, fn)(gp.h, 0, slots, qd, out, update, check=False)
    torch.cuda.synchronize()
    if fn.endswith("_static"):
        FREE_SEEN.append((before, torch.cuda.mem_get_info()[0]))
    return rc, out.cpu().numpy()


def assert_nothing_allocated():
    assert FREE_SEEN and all(a == b for a, b in FREE_SEEN), FREE_SEEN


def need_bytes(n_units, G, max_n, update):
    """Scratch bytes of one call, from the formula the header states."""
    r = lambda x: (x + 255) // 256 * 256
    C = (max_n + 15) // 16 + 1
    b = r(4 * n_units * G) + r(4 * n_units * (C // 8 + 2) * (128 * G + 16))
    return b + (64 * G * n_units * C if update else 0)


@pytest.mark.parametrize("pb", [4096, 3584, 8192])
def test_static_matches_pool_scratch_on_consecutive_calls(pb):
    """4 KB pages (the kernel for any geometry), 3.5 KB pages (16 / 32 tokens,
    the paged kernel) and 8 KB pages (32 / 64 tokens, the paged kernel as
    four CTAs of 4 warps per SM)."""
    FREE_SEEN.clear()
    cfg = cfg_of(page_bytes=pb, **(dict(tokens_per_hi_page=32, tokens_per_lo_page=64) if pb == 8192 else {}))
    lens = [600, 257, 1100]
    n = sum(lens)
    k = workloads.random_fp16((n, 2, 128), 70, scale=1.5)
    v = workloads.random_fp16((n, 2, 128), 71)
    S = workloads.given_scores(n, 2, seed=72)
    with GPool(cfg) as ga, GPool(cfg) as gb:
        ga.prompt(0, [0, 1, 2], lens, k, v, scores_in=S)
        gb.prompt(0, [0, 1, 2], lens, k, v, scores_in=S)
        # two calls in a row with score updates, then one over a subset without
        for step, (slots, update) in enumerate([([0, 1, 2], True), ([0, 1, 2], True), ([2, 0], False)]):
            q = workloads.random_fp16((len(slots), 8, 128), 700 + step, scale=2.0)
            rc_a, ref = attend(ga, "dkv_decode_attention", slots, q, update)
            rc_b, out = attend(gb, "dkv_decode_attention_static", slots, q, update)
            assert rc_a == 0 and rc_b == 0, (rc_a, rc_b)
            assert np.isfinite(out).all()
            ok, worst = parity.within(out.astype(np.float64), ref.astype(np.float64), ATT_ATOL, ATT_RTOL)
            assert ok, (step, worst)
        assert ga.status()["error"] == 0 and gb.status()["error"] == 0
        sa, sb = ga.snapshot(), gb.snapshot()
        assert (sa["req_state"] == sb["req_state"]).all()
        assert (sa["head_counts"] == sb["head_counts"]).all()
        for i in range(3):
            for h in range(2):
                for a, b in zip(stored(sa, (0, i, h), ga.t_hi, ga.t_lo, 4, np.float32),
                                stored(sb, (0, i, h), gb.t_hi, gb.t_lo, 4, np.float32)):
                    ok, worst = parity.within(b.astype(np.float64), a.astype(np.float64), 1e-6, 1e-4)
                    assert ok, worst
    assert_nothing_allocated()


def test_static_against_oracle():
    """Two static calls in a row with score updates, each against the
    oracle's fp64 attention over the same state (outputs and updated scores),
    so that a fault shared by both GPU entry points cannot pass unseen."""
    FREE_SEEN.clear()
    cfg = cfg_of(page_bytes=3584)
    lens = [900, 333, 64]
    n = sum(lens)
    k = workloads.random_fp16((n, 2, 128), 90, scale=1.5)
    v = workloads.random_fp16((n, 2, 128), 91)
    S = workloads.given_scores(n, 2, seed=92)
    op = oracle.Pool(cfg)
    with GPool(cfg) as gp:
        gp.prompt(0, [0, 1, 2], lens, k, v, scores_in=S)
        for step in range(2):
            load_into(op, gp.snapshot())
            q = workloads.random_fp16((3, 8, 128), 900 + step, scale=2.0)
            rc, out = attend(gp, "dkv_decode_attention_static", [0, 1, 2], q, True)
            assert rc == 0
            rc, ref = op.attention(0, [0, 1, 2], q, update_scores=True)
            assert rc == 0
            ok, worst = parity.within(out.astype(np.float64), ref, ATT_ATOL, ATT_RTOL)
            assert ok, (step, worst)
            gs, os_ = gp.snapshot(), op.snapshot()
            assert (gs["req_state"] == os_["req_state"]).all()
            for i in range(3):
                for h in range(2):
                    for a, b in zip(stored(gs, (0, i, h), gp.t_hi, gp.t_lo, 4, np.float32),
                                    stored(os_, (0, i, h), gp.t_hi, gp.t_lo, 4, np.float32)):
                        ok, worst = parity.within(a.astype(np.float64), b.astype(np.float64), 1e-6, 1e-4)
                        assert ok, worst
    assert_nothing_allocated()


def test_static_limit_counts_pruned_tokens():
    """The size limit follows each request's length N, pruned tokens
    included: 64 requests of 4096 tokens with every token outside the recent
    window pruned store 64 tokens a head, yet the call is refused, as the
    header's formula with max_n = N says."""
    import differentiated_kv_cache_gb300 as dkv
    R, L, H, G = 64, 4096, 8, 8
    cfg = cfg_of(n_kv_heads=H, group_size=G, max_requests=R, max_seq_len=L, page_bytes=3584,
                 n_pages=R * H * (L // 16 + 2))
    assert need_bytes(R * H, G, L, False) > dkv.DKV_ATTN_STATIC_SCRATCH_BYTES
    assert need_bytes(R * H, G, 64, True) <= dkv.DKV_ATTN_STATIC_SCRATCH_BYTES
    n = R * L
    k = np.zeros((n, H, 128), np.float16)
    S = np.zeros((n, H), np.float32)                 # importance 0: pruned outside the window
    with GPool(cfg) as gp:
        gp.prompt(0, list(range(R)), [L] * R, k, k, scores_in=S)
        st = gp.status()
        assert st["hi_tokens"] == R * H * 64 and st["lo_tokens"] == 0, st
        q = workloads.random_fp16((R, H * G, 128), 95)
        for update in (False, True):
            rc, out = attend(gp, "dkv_decode_attention_static", list(range(R)), q, update)
            assert rc == dkv.DKV_ERR_SCRATCH, rc
            assert np.isnan(out).all()


def test_static_rejects_calls_beyond_the_array():
    """1024 short requests of 8 KV heads with G = 8 need more than 64 MiB of
    partials: the call is refused on the host with nothing queued; half of
    them fit and match the pool-scratch entry point."""
    import differentiated_kv_cache_gb300 as dkv
    FREE_SEEN.clear()
    R, L, H, G = 1024, 40, 8, 8
    cfg = cfg_of(n_kv_heads=H, group_size=G, max_requests=R, max_seq_len=64, n_pages=R * H * 5)
    assert need_bytes(R * H, G, L, False) > dkv.DKV_ATTN_STATIC_SCRATCH_BYTES
    assert need_bytes(R // 2 * H, G, L, True) <= dkv.DKV_ATTN_STATIC_SCRATCH_BYTES
    n = R * L
    k = workloads.random_fp16((n, H, 128), 80)
    v = workloads.random_fp16((n, H, 128), 81)
    S = workloads.given_scores(n, H, seed=82)
    slots = list(range(R))
    with GPool(cfg) as ga, GPool(cfg) as gb:
        ga.prompt(0, slots, [L] * R, k, v, scores_in=S)
        gb.prompt(0, slots, [L] * R, k, v, scores_in=S)
        before = gb.snapshot(pages=False)
        q = workloads.random_fp16((R, H * G, 128), 83)
        for update in (False, True):
            rc, out = attend(gb, "dkv_decode_attention_static", slots, q, update)
            assert rc == dkv.DKV_ERR_SCRATCH, rc
            assert np.isnan(out).all()
        assert dkv.dkv_strerror(dkv.DKV_ERR_SCRATCH) != "unknown error"
        after = gb.snapshot(pages=False)
        for key in ("free_list", "table", "head_counts", "req_state"):
            assert (before[key] == after[key]).all(), key
        assert gb.status()["error"] == 0
        half = slots[: R // 2]
        for step in range(2):
            qh = q[: R // 2] if step == 0 else workloads.random_fp16((R // 2, H * G, 128), 84)
            rc_a, ref = attend(ga, "dkv_decode_attention", half, qh, True)
            rc_b, out = attend(gb, "dkv_decode_attention_static", half, qh, True)
            assert rc_a == 0 and rc_b == 0, (rc_a, rc_b)
            ok, worst = parity.within(out.astype(np.float64), ref.astype(np.float64), ATT_ATOL, ATT_RTOL)
            assert ok, (step, worst)
        assert (ga.snapshot(pages=False)["req_state"] == gb.snapshot(pages=False)["req_state"]).all()
    assert_nothing_allocated()

"""Churn of the circular free list (DiffKV, Memory management: circular free
page list, bidirectional page table, prompt and generation workflows) under
dynamic arrivals and completions.

CPU: the oracle alone through hundreds of ticks, the memory-management
invariants after every operation (the free list's live region and the
tables together a permutation of the pool, hi and lo regions apart, page
counts matching token counts), both counters wrapping the pool several times,
and every page back in the list at the end.

GPU: the same traffic through the C ABI; before every operation the oracle
takes over the GPU's state, both run it, and the states must be identical.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tests import pagefmt
from tests.churn import Churn

H, G = 2, 4


def churn_cfg(**over):
    cfg = dict(n_layers=1, n_kv_heads=H, group_size=G, head_dim=128, page_bytes=3584, n_pages=400,
               max_requests=6, max_seq_len=800, tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=1,
               alpha_h=2.0, alpha_l=0.25, recent_window=16, obs_window=32, prompt_grant_slack=1,
               reclaim_in_decode=1)
    cfg.update(over)
    return cfg


def prompt_inputs(n0: int, seed: int):
    k = workloads.random_fp16((n0, H, 128), seed, scale=1.5)
    v = workloads.random_fp16((n0, H, 128), seed + 1)
    S = workloads.given_scores(n0, H, seed=seed + 2, scale=0.2)
    return k, v, S


def step_inputs(n: int, tick: int):
    return (workloads.random_fp16((n, H, 128), 70000 + tick), workloads.random_fp16((n, H, 128), 80000 + tick),
            workloads.random_fp16((n, H * G, 128), 90000 + tick, scale=2.0))


# the three-tier pool (mid tier K8V2; its pages in the one-way part of each row)
MID = dict(mid_enabled=1, alpha_m=0.8, tokens_per_mid_page=16, prompt_grant_slack=2)


@pytest.mark.parametrize("reclaim,mid", [(1, 0), (0, 0), (1, 1)])
def test_oracle_churn_invariants(reclaim, mid):
    cfg = churn_cfg(reclaim_in_decode=reclaim, **(MID if mid else {}))
    op = oracle.Pool(cfg)
    ch = Churn(seed=3 + reclaim + 5 * mid, max_requests=cfg["max_requests"], n_kv_heads=H, t_hi=op.t_hi,
               slack=cfg["prompt_grant_slack"], tiers=3 if mid else 2)
    n_ops = 0
    for tick in range(400):
        free = int(op.pointers[1] - op.pointers[0])
        kn, vn, q = None, None, None
        for o in ch.tick(free):
            if o[0] == "prompt":
                k, v, S = prompt_inputs(o[2], o[3])
                assert op.prompt(0, [o[1]], [o[2]], k, v, scores_in=S) == 0
            elif o[0] == "decode":
                kn, vn, q = step_inputs(len(o[1]), tick)
                assert op.decode(0, o[1], kn, vn) == 0
            elif o[0] == "attend":
                rc, _ = op.attention(0, o[1], q, update_scores=True)
                assert rc == 0
            else:
                assert op.free_request(o[1]) == 0
            n_ops += 1
            pagefmt.check_invariants(op.snapshot(), op.t_hi, op.t_lo, cfg["n_pages"], reclaim=bool(reclaim),
                                     table_len=op.table_len, t_mid=op.t_mid)
    start, end = (int(x) for x in op.pointers)
    assert start >= 3 * cfg["n_pages"] and end >= 4 * cfg["n_pages"], (start, end)
    for s in sorted(ch.active):
        assert op.free_request(s) == 0
    snap = op.snapshot()
    assert int(snap["pointers"][1] - snap["pointers"][0]) == cfg["n_pages"] and (snap["table"] == -1).all()
    print(f"{ch.n_arrived} requests, {n_ops} operations, list start {start} end {end} "
          f"({end // cfg['n_pages']} wraps)")


@pytest.mark.gpu
@pytest.mark.parametrize("mid", [0, 1])
def test_gpu_churn_bit_exact(mid):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiated_kv_cache_gb300 as dkv
    from tests import parity
    from tests.gpu_pool import GPool, load_into
    dkv.build.build()
    dkv.load()
    cfg = churn_cfg(**(MID if mid else {}))
    op = oracle.Pool(cfg)
    with GPool(cfg) as gp:
        ch = Churn(seed=11 + mid, max_requests=cfg["max_requests"], n_kv_heads=H, t_hi=gp.t_hi,
                   slack=cfg["prompt_grant_slack"], tiers=3 if mid else 2)
        q = None
        for tick in range(300):
            free = gp.status()["free_pages"]
            for o in ch.tick(free):
                load_into(op, gp.snapshot())
                if o[0] == "prompt":
                    k, v, S = prompt_inputs(o[2], o[3])
                    gp.prompt(0, [o[1]], [o[2]], k, v, scores_in=S)
                    assert op.prompt(0, [o[1]], [o[2]], k, v, scores_in=S) == 0
                elif o[0] == "decode":
                    kn, vn, q = step_inputs(len(o[1]), tick)
                    gp.decode(0, o[1], kn, vn)
                    assert op.decode(0, o[1], kn, vn) == 0
                elif o[0] == "attend":
                    gp.attention(0, o[1], q, update=True)
                    continue          # scores: fp32 on the GPU against fp64 (compared elsewhere)
                else:
                    gp.free(o[1])
                    assert op.free_request(o[1]) == 0
                assert gp.status()["error"] == 0
                parity.compare_states(gp.snapshot(), op.snapshot(), gp.t_hi, gp.t_lo, cfg["n_pages"],
                                      cfg["page_bytes"], table_len=gp.table_len, t_mid=gp.t_mid)
        st = gp.status()
        assert st["list_start"] >= 3 * cfg["n_pages"], st
        print(f"{ch.n_arrived} requests; list start {st['list_start']} end {st['list_end']}")

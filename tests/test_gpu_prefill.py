"""GPU parity of the prompt's own causal attention (dkv_prefill_attention) and
of the PROMPT compaction that takes that attention's observation-row
log-sum-exps instead of its own pass over the keys
(dkv_compact_step_prefilled), against the oracle's fp64 attention and fp64
scores on the same seeded inputs.

- Ragged batches (1 to 700 tokens: single tokens, prompts shorter than the
  32 observation rows, lengths one either side of the 64-row query tiles and
  64-key key tiles) and workload-shaped layers (outlier channels, per-head
  key temperature, heavy hitters, G = 1 .. 8): every output element and every
  observation row's log-sum-exp, -inf for rows before the prompt's start.
- The prefilled compaction: scores within the score tolerance of the fp64
  scores, and the oracle fed the GPU's own scores reproduces the GPU state
  bit for bit.
- The llama8b batch at full size (32 x 4096 tokens, 32 query heads): sampled
  rows (tile edges, the middle, every observation row) of three requests over
  every head, then the prefilled compaction of the whole batch.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from tests import parity
from tests.gpu_pool import GPool

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

# Output: |gpu - ref| <= PF_ATOL + PF_RTOL |ref| elementwise against fp64.
# Sources of error, relative to the largest |v| the row averages: fp32
# accumulation of the fp16 logits (at most a few 1e-6 in base-2 units on
# these inputs, which moves each probability by that factor), ex2.approx
# (2 ulp), the fp16 pair that carries a probability into the value product
# (2^-22) and fp32 accumulation of up to 4096 terms (sqrt growth, ~1e-5 at
# most); |v| stays below ~40 with the outlier channels, so 2e-4 absolute
# holds each row with a margin of several times, and the relative term covers
# rows dominated by one large value.
PF_ATOL, PF_RTOL = 2e-4, 2e-4
# Log-sum-exp (base 2): the logit error above plus log2f and the fp32 sum.
LSE_ATOL, LSE_RTOL = 5e-5, 1e-6
# Scores from the given log-sum-exps: the same tolerance as the scores the
# score pass computes with its own (fp32 tensor-core logits, exp2), since the
# log-sum-exps carry the same fp32 logit error.
SC_ATOL, SC_RTOL = 1e-6, 5e-5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiated_kv_cache_gb300 as dkv
    dkv.build.build()
    dkv.load()


def _dkv():
    import differentiated_kv_cache_gb300 as dkv
    return dkv


def _cfg(H, G, lens, **over):
    c = dict(n_layers=1, n_kv_heads=H, group_size=G, head_dim=128, page_bytes=4096, n_pages=8192,
             max_requests=len(lens), max_seq_len=max(lens) + 8, tokens_per_hi_page=0, tokens_per_lo_page=0,
             lo_enabled=1, alpha_h=2.0, alpha_l=0.25, recent_window=64, obs_window=32, prompt_grant_slack=1,
             reclaim_in_decode=1)
    c.update(over)
    return c


def gpu_prefill(gp, lens, q, k, v, want_lse=True):
    """dkv_prefill_attention on the pool's device; returns (out, lse_obs)."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    R, Hq = len(lens), q.shape[1]
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((R, Hq, 32), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    _dkv().dkv_prefill_attention(gp.h, lens, dev(q), dev(k), dev(v), out, lse)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (lse.cpu().numpy() if want_lse else None)


def oracle_prefill(lens, q, k, v, H, G):
    """fp64 attention of every request and KV head: out [T, Hq, 128], lse2 [T, Hq]."""
    T = int(np.sum(lens))
    out = np.zeros((T, H * G, 128))
    lse2 = np.zeros((T, H * G))
    t0 = 0
    for n0 in lens:
        for h in range(H):
            o, l2 = oracle.prefill_attention(q[t0:t0 + n0, h * G:(h + 1) * G], k[t0:t0 + n0, h],
                                             v[t0:t0 + n0, h])
            out[t0:t0 + n0, h * G:(h + 1) * G] = o
            lse2[t0:t0 + n0, h * G:(h + 1) * G] = l2
        t0 += n0
    return out, lse2


def check_lse_obs(lse_obs, lse2, lens):
    """Every observation row: the fp64 log-sum-exp at its position, -inf before the prompt."""
    t0 = 0
    worst = -np.inf
    for i, n0 in enumerate(lens):
        for o in range(32):
            p = n0 - 32 + o
            if p < 0:
                assert np.isneginf(lse_obs[i, :, o]).all(), (i, o)
                continue
            ok, w = parity.within(lse_obs[i, :, o].astype(np.float64), lse2[t0 + p], LSE_ATOL, LSE_RTOL)
            assert ok, (i, o, w)
            worst = max(worst, w)
        t0 += n0
    return worst


def _random_case(H, G, lens, seed):
    T = int(np.sum(lens))
    q = workloads.random_fp16((T, H * G, 128), seed, scale=1.5)
    k = workloads.random_fp16((T, H, 128), seed + 1, scale=1.5)
    v = workloads.random_fp16((T, H, 128), seed + 2)
    return q, k, v


CASES = {
    "ragged_g4": (2, 4, [1, 5, 31, 32, 33, 63, 64, 65, 127, 200]),
    "g8": (1, 8, [300, 2]),
    "g1": (3, 1, [129]),
}
WORKLOAD_CASES = {
    "tiny": ("tiny", None, None),                       # outlier channels, 512 and 700 tokens
    "qwen7b": ("qwen7b", [0, 1], 1100),                 # G = 7, skewed key temperature
    "llama70b": ("llama70b", [0], 1000),                # G = 8, heavy hitters
}


def _case(name):
    if name in CASES:
        H, G, lens = CASES[name]
        q, k, v = _random_case(H, G, lens, 900 + len(lens))
        return H, G, list(lens), q, k, v
    wname, reqs, max_len = WORKLOAD_CASES[name]
    w = workloads.WORKLOADS[wname]
    inp = workloads.prefill_inputs(wname, 0, reqs, max_len)
    return w.n_kv_heads, w.group_size, [int(x) for x in inp["lens"]], inp["q"], inp["k"], inp["v"]


@pytest.mark.parametrize("name", list(CASES) + list(WORKLOAD_CASES))
def test_prefill_attention_parity(name):
    H, G, lens, q, k, v = _case(name)
    with GPool(_cfg(H, G, lens)) as gp:
        out, lse_obs = gpu_prefill(gp, lens, q, k, v)
        assert gp.status()["error"] == 0
    ref, lse2 = oracle_prefill(lens, q, k, v, H, G)
    assert not np.isnan(out).any()
    ok, worst = parity.within(out.astype(np.float64), ref, PF_ATOL, PF_RTOL)
    err = np.abs(out - ref).max()
    print(f"{name}: {len(lens)} prompts, max |out err| {err:.3e}, tolerance excess {worst:.3e}")
    assert ok, worst
    lw = check_lse_obs(lse_obs, lse2, lens)
    print(f"{name}: log-sum-exp tolerance excess {lw:.3e}")


def test_prefill_attention_without_lse_and_error_codes():
    H, G, lens = 2, 4, [70, 3]
    q, k, v = _random_case(H, G, lens, 950)
    dkv = _dkv()
    with GPool(_cfg(H, G, lens)) as gp:
        out, _ = gpu_prefill(gp, lens, q, k, v, want_lse=False)
        ref, _ = oracle_prefill(lens, q, k, v, H, G)
        assert parity.within(out.astype(np.float64), ref, PF_ATOL, PF_RTOL)[0]
        qd, kd, vd = (torch.from_numpy(a).cuda() for a in (q, k, v))
        o = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
        E = dkv.DKV_ERR_ARG
        assert dkv.dkv_prefill_attention(gp.h, [], qd, kd, vd, o, check=False) == E
        assert dkv.dkv_prefill_attention(gp.h, [0, 3], qd, kd, vd, o, check=False) == E
        assert dkv.dkv_prefill_attention(gp.h, [max(lens) + 9, 3], qd, kd, vd, o, check=False) == E
        qm = torch.zeros(q.size + 8, dtype=torch.float16, device="cuda")[4:4 + q.size].view(q.shape)
        assert dkv.dkv_prefill_attention(gp.h, lens, qm, kd, vd, o, check=False) == E
        assert gp.status()["error"] == 0


def _prefilled_compaction(gp, slots, lens, q, k, v, q_obs):
    """Prefill for the log-sum-exps, then the prefilled PROMPT compaction."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    _, lse_obs = gpu_prefill(gp, lens, q, k, v)
    so = torch.zeros((int(np.sum(lens)), gp.cfg["n_kv_heads"]), dtype=torch.float32, device="cuda")
    _dkv().dkv_compact_step_prefilled(gp.h, 0, slots, lens, dev(k), dev(v), dev(q_obs),
                                      torch.from_numpy(lse_obs).cuda(), so)
    torch.cuda.synchronize()
    return so.cpu().numpy()


def _fp64_scores(k, q_obs, lens, H, G):
    S64 = np.zeros((int(np.sum(lens)), H))
    t0 = 0
    for i, n0 in enumerate(lens):
        for h in range(H):
            S64[t0:t0 + n0, h] = oracle.unit_scores(k[t0:t0 + n0, h], q_obs[i][:, h * G:(h + 1) * G])
        t0 += n0
    return S64


@pytest.mark.parametrize("name", ["tiny", "qwen7b", "ragged_g8"])
def test_prefilled_compaction_parity(name):
    if name == "ragged_g8":
        H, G, lens = 2, 8, [20, 31, 32, 33, 100, 257, 640]
        q, k, v = _random_case(H, G, lens, 960)
        q_obs = np.zeros((len(lens), 32, H * G, 128), np.float16)
        t0 = 0
        for i, n0 in enumerate(lens):
            m = min(n0, 32)
            q_obs[i, 32 - m:] = q[t0 + n0 - m:t0 + n0]
            t0 += n0
        lo_enabled = 1
    else:
        wname, reqs, max_len = WORKLOAD_CASES[name]
        w = workloads.WORKLOADS[wname]
        inp = workloads.prefill_inputs(wname, 0, reqs, max_len)
        H, G, lens = w.n_kv_heads, w.group_size, [int(x) for x in inp["lens"]]
        q, k, v, q_obs = inp["q"], inp["k"], inp["v"], inp["q_obs"]
        lo_enabled = w.lo_enabled
    cfg = _cfg(H, G, lens, lo_enabled=lo_enabled)
    slots = list(range(len(lens)))[::-1]
    with GPool(cfg) as gp:
        so = _prefilled_compaction(gp, slots, lens, q, k, v, q_obs)
        assert gp.status()["error"] == 0
        gsnap = gp.snapshot()
    S64 = _fp64_scores(k, q_obs, lens, H, G)
    ok, worst = parity.within(so.astype(np.float64), S64, SC_ATOL, SC_RTOL)
    rel = np.abs(so - S64) / np.maximum(S64, 1e-30)
    print(f"{name}: score max rel err {rel.max():.3e}, tolerance excess {worst:.3e}")
    assert ok, worst
    op = oracle.Pool(cfg)
    assert op.prompt(0, slots, lens, k, v, scores_in=so) == 0
    parity.compare_states(gsnap, op.snapshot(), gp.t_hi, gp.t_lo, cfg["n_pages"], cfg["page_bytes"])


def test_prefilled_compaction_state_errors():
    H, G, lens = 1, 4, [40]
    q, k, v = _random_case(H, G, lens, 970)
    q_obs = q[None, 8:40]
    dkv = _dkv()
    with GPool(_cfg(H, G, lens)) as gp:
        _prefilled_compaction(gp, [0], lens, q, k, v, q_obs)
        kd, vd, qo = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (k, v, q_obs))
        lse = torch.zeros((1, G, 32), dtype=torch.float32, device="cuda")
        assert dkv.dkv_compact_step_prefilled(gp.h, 0, [0], lens, kd, vd, qo, lse, check=False) == \
            dkv.DKV_ERR_STATE
        assert dkv.dkv_compact_step_prefilled(gp.h, 1, [0], lens, kd, vd, qo, lse, check=False) == \
            dkv.DKV_ERR_ARG
        assert dkv.dkv_compact_step_prefilled(gp.h, 0, [0], lens, kd, vd, qo, None, check=False) == \
            dkv.DKV_ERR_ARG
        assert gp.status()["error"] == 0


def test_prefill_llama8b_full_size():
    name = "llama8b"
    w = workloads.WORKLOADS[name]
    H, G = w.n_kv_heads, w.group_size
    inp = workloads.prefill_inputs(name, 0)
    lens = [int(x) for x in inp["lens"]]
    slots = list(range(w.n_requests))
    cfg = w.pool_config()
    with GPool(cfg) as gp:
        out, lse_obs = gpu_prefill(gp, lens, inp["q"], inp["k"], inp["v"])
        assert not np.isnan(out).any()
        # sampled rows of three requests over every head
        pos = np.array([0, 1, 62, 63, 64, 65, 127, 128, 1000, 2047, 2048, 3071, 4000, 4031, 4063, 4064, 4095])
        worst = -np.inf
        for i in (0, 13, 31):
            t0 = int(np.sum(lens[:i]))
            for h in range(H):
                ref, l2 = oracle.prefill_rows(pos, inp["q"][t0 + pos, h * G:(h + 1) * G], inp["k"][t0:t0 + 4096, h],
                                              inp["v"][t0:t0 + 4096, h])
                ok, wo = parity.within(out[t0 + pos, h * G:(h + 1) * G].astype(np.float64), ref, PF_ATOL, PF_RTOL)
                assert ok, (i, h, wo)
                worst = max(worst, wo)
                obs = np.arange(4064, 4096)
                _, lo = oracle.prefill_rows(obs, inp["q"][t0 + obs, h * G:(h + 1) * G], inp["k"][t0:t0 + 4096, h],
                                            inp["v"][t0:t0 + 4096, h])
                ok, wl = parity.within(lse_obs[i, h * G:(h + 1) * G].T.astype(np.float64), lo, LSE_ATOL, LSE_RTOL)
                assert ok, (i, h, wl)
        print(f"{name}: sampled rows within tolerance (excess {worst:.3e})")
        # the prefilled compaction of the whole batch
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        so = torch.zeros((sum(lens), H), dtype=torch.float32, device="cuda")
        _dkv().dkv_compact_step_prefilled(gp.h, 0, slots, lens, dev(inp["k"]), dev(inp["v"]), dev(inp["q_obs"]),
                                          torch.from_numpy(lse_obs).cuda(), so)
        torch.cuda.synchronize()
        so = so.cpu().numpy()
        assert gp.status()["error"] == 0
        gsnap = gp.snapshot()
    from tests.test_gpu_full_parity import _fp64_scores as full_scores
    S64 = full_scores(inp, H, G, lens)
    ok, worst = parity.within(so.astype(np.float64), S64, SC_ATOL, SC_RTOL)
    print(f"{name}: prefilled scores, tolerance excess {worst:.3e}")
    assert ok, worst
    op = oracle.Pool(cfg)
    assert op.prompt(0, slots, lens, inp["k"], inp["v"], scores_in=so) == 0
    parity.compare_states(gsnap, op.snapshot(), gp.t_hi, gp.t_lo, cfg["n_pages"], cfg["page_bytes"])

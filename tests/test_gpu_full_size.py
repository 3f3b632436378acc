"""GPU parity at the model-shaped workloads' full sizes, in the launch
configuration the benchmark times (every head of the workload in one call):
a prompt compact_step with scores computed from the observation queries, one
generation-phase step, then decode attention with score updates. The oracle's
fp64 attention of sampled heads runs over the GPU pool's own pages (copied into
an oracle pool), so the check covers the attention kernel's range partition,
its epilogue and the score update at the sizes they are timed at, one head at
a time."""
import numpy as np
import pytest

import oracle
import workloads
from tests import parity
from tests.gpu_pool import GPool, stored

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ATT_ATOL, ATT_RTOL = 1e-3, 2e-3       # attention output (fp64 reference)
SC_ATOL, SC_RTOL = 1e-6, 1e-4         # updated scores: one fp32 add of a probability


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import differentiated_kv_cache_gb300 as dkv
    dkv.build.build()
    dkv.load()


def sampled_heads(R, H, n=10):
    """First and last heads, heads around every quarter of the head order
    (where attention ranges of neighbouring heads meet), and a spread of
    others: (request, kv head) pairs."""
    units = sorted({0, 1, R * H - 1, R * H // 4, R * H // 2, 3 * R * H // 4, R * H // 2 + 1,
                    *np.linspace(0, R * H - 1, n).astype(int).tolist()})
    return [(u // H, u % H) for u in units]


@pytest.mark.parametrize("name", ["llama8b", "llama70b"])
def test_full_size_attention_and_score_update(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.prompt_inputs(name, 0)
    dec = workloads.decode_inputs(name, 0)
    cfg = w.pool_config()
    R, H, G = w.n_requests, w.n_kv_heads, w.group_size
    slots = list(range(R))
    lens = [int(x) for x in inp["lens"]]
    with GPool(cfg) as gp:
        gp.prompt(0, slots, lens, inp["k"], inp["v"], inp["q_obs"])
        gp.decode(0, slots, dec["k"], dec["v"])
        before = gp.snapshot()
        out = gp.attention(0, slots, dec["q"], update=True)
        after = gp.snapshot(pages=True)
        assert gp.status()["error"] == 0
        t_hi, t_lo = gp.t_hi, gp.t_lo
    op = oracle.Pool(cfg)
    for key in ("pages", "free_list", "table", "head_counts", "req_state", "pointers"):
        getattr(op, key)[...] = before[key]
    worst_att = worst_sc = 0.0
    bad = []
    for i, h in sampled_heads(R, H):
        q_group = dec["q"][i, h * G:(h + 1) * G]
        ref, pm = op.unit_attention(0, i, h, q_group)
        got = out[i, h * G:(h + 1) * G].astype(np.float64)
        r = np.abs(got - ref) / (ATT_ATOL + ATT_RTOL * np.abs(ref))
        k = np.unravel_index(int(r.argmax()), r.shape)
        cnt = before["head_counts"][0, i, h]
        print(f"{name} head ({i},{h}) hi {cnt[0]} lo {cnt[1]}: attention err/tol {r.max():.3f} at {k} "
              f"(gpu {got[k]:.6f}, ref {ref[k]:.6f}), |ref| max {np.abs(ref).max():.3f}")
        if r.max() > 1.0:
            bad.append(("attention", i, h, float(r.max())))
        worst_att = max(worst_att, float(r.max()))
        old = np.concatenate(stored(before, (0, i, h), t_hi, t_lo, 4, np.float32)).astype(np.float64)
        new = np.concatenate(stored(after, (0, i, h), t_hi, t_lo, 4, np.float32)).astype(np.float64)
        assert new.shape == pm.shape
        rs = np.abs(new - old - pm) / (SC_ATOL + SC_RTOL * np.abs(old + pm))
        if rs.max() > 1.0:
            bad.append(("score", i, h, float(rs.max())))
        worst_sc = max(worst_sc, float(rs.max()))
    print(f"{name}: {len(sampled_heads(R, H))} heads, attention max err/tolerance {worst_att:.3f}, "
          f"scores {worst_sc:.3f}")
    assert not bad, bad

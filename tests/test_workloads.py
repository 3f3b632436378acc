"""The seeded input recipe: shapes, determinism and the structure each
workload is stated to carry (outlier channels, per-head low-rank bias,
heavy hitters, per-head key temperature, ragged prompt lengths)."""
import dataclasses

import numpy as np
import pytest

import workloads


def test_shapes_and_subset_draws_are_the_full_draw_rows():
    full = workloads.prompt_inputs("tiny", 0)
    w = workloads.WORKLOADS["tiny"]
    assert list(full["lens"]) == [512, 700]
    assert full["k"].shape == (1212, w.n_kv_heads, 128) and full["k"].dtype == np.float16
    assert full["q_obs"].shape == (2, 32, w.n_q_heads, 128)
    one = workloads.prompt_inputs("tiny", 0, requests=[1])
    assert (one["k"] == full["k"][512:]).all() and (one["v"] == full["v"][512:]).all()
    assert (one["q_obs"][0] == full["q_obs"][1]).all()
    again = workloads.prompt_inputs("tiny", 0)
    assert all((again[x] == full[x]).all() for x in ("k", "v", "q_obs"))
    other = workloads.prompt_inputs("tiny", 1)
    assert not (other["k"] == full["k"]).all()
    d = workloads.decode_inputs("tiny", 3)
    d1 = workloads.decode_inputs("tiny", 3, requests=[1])
    assert d["q"].shape == (2, w.n_q_heads, 128) and (d1["k"][0] == d["k"][1]).all()


def test_outlier_channels_are_scaled():
    w = workloads.WORKLOADS["tiny"]
    st = workloads.head_structure(w, 0)
    k = workloads.prompt_inputs("tiny", 0)["k"].astype(np.float32)
    for h in range(w.n_kv_heads):
        sd = k[:, h, :].std(axis=0)
        out = np.zeros(128, bool)
        out[st.outlier_idx[h]] = True
        ratio = sd[out].mean() / sd[~out].mean()
        assert 6.5 < ratio < 9.5, ratio


def test_ragged_lengths_and_temperature_of_qwen7b():
    w = workloads.WORKLOADS["qwen7b"]
    lens = workloads.prompt_lengths(w, 0)
    assert lens.shape == (128,) and lens.min() >= 1024 and lens.max() <= 16384
    assert lens.max() - lens.min() > 8000                      # spread over the range
    st = workloads.head_structure(w, 0)
    assert st.temp.shape == (4,) and (st.temp >= 2 ** 0.5).all() and (st.temp <= 2 ** 3.5).all()


def test_low_rank_bias_tilts_the_queries_toward_their_head():
    """A query of head group h lines up better with group h's key bias
    directions than with another group's."""
    w = workloads.WORKLOADS["llama8b"]
    st = workloads.head_structure(w, 0)
    q = workloads.decode_inputs("llama8b", 0)["q"].astype(np.float32)   # [32, 32, 128]
    own, other = [], []
    for hq in range(w.n_q_heads):
        h = hq // w.group_size
        basis = [np.linalg.qr(st.bias_k[x])[0] for x in (h, (h + 1) % w.n_kv_heads)]
        proj = [np.linalg.norm(q[:, hq, :] @ b, axis=1).mean() for b in basis]
        own.append(proj[0])
        other.append(proj[1])
    assert np.mean(own) > 1.2 * np.mean(other)


def test_heavy_hitters_raise_the_mean_query_logit(monkeypatch):
    """The llama70b structure on a short prompt: 2% of the keys outside the
    recent window gain +3 sigma of logit against the group's mean
    observation query."""
    w = dataclasses.replace(workloads.WORKLOADS["llama70b"], name="heavy", n_requests=1, prompt_len=3000)
    monkeypatch.setitem(workloads.WORKLOADS, "heavy", w)
    base = dataclasses.replace(w, name="plain", heavy_frac=0.0)
    monkeypatch.setitem(workloads.WORKLOADS, "plain", base)
    hv = workloads.prompt_inputs("heavy", 0)
    pl = workloads._rng  # the same streams: draw the plain keys under the heavy workload's name
    monkeypatch.setattr(workloads, "_rng", lambda name, seed, role, step=0: pl("heavy", seed, role, step))
    pk = workloads.prompt_inputs("plain", 0)["k"].astype(np.float32)
    hk = hv["k"].astype(np.float32)
    moved = np.abs(hk - pk).max(axis=2) > 1e-2                       # [n, Hkv]
    eligible = 3000 - w.recent_window
    for h in range(w.n_kv_heads):
        pos = np.nonzero(moved[:, h])[0]
        assert len(pos) == round(0.02 * eligible) and pos.max() < eligible
        mean_q = hv["q_obs"][0][:, h * w.group_size:(h + 1) * w.group_size].astype(np.float32) \
            .reshape(-1, 128).mean(axis=0)
        base = pk[:, h, :] @ mean_q / np.sqrt(128)
        boost = (hk[pos, h, :] - pk[pos, h, :]) @ mean_q / np.sqrt(128)
        assert boost.mean() == pytest.approx(3.0 * base.std(), rel=0.02)

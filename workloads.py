"""Seeded synthetic workloads for differentiated KV compaction.

This module only draws random inputs with the shapes and structure of the
workloads (model-shaped KV heads, outlier channels, low-rank bias, heavy
hitters, skewed per-head temperature). It holds none of the compaction
method's arithmetic, and both the oracle tests and the GPU path take their
inputs from it.

All arrays are numpy; fp16 data is produced by rounding float32 normals to
binary16 (numpy's conversion is round-to-nearest-even). The generator is
numpy's PCG64 (``np.random.default_rng``), seeded per (workload, seed, role,
step) so that every input can be regenerated independently.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field, asdict

import numpy as np

HEAD_DIM = 128
OBS_WINDOW = 32


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    n_kv_heads: int
    group_size: int
    n_requests: int
    prompt_len: int | tuple[int, int]       # fixed, or (lo, hi) uniform integer range
    decode_steps: int
    n_pages: int
    alpha_h: float = 2.0
    alpha_l: float = 0.25
    lo_enabled: int = 1
    recent_window: int = 64
    outlier_channels: int = 4
    outlier_scale: float = 8.0
    bias_rank: int = 0                       # per-KV-head low-rank key/value bias
    bias_std: float = 0.35                    # std of the bias basis entries
    heavy_frac: float = 0.0                  # fraction of heavy-hitter keys
    heavy_sigma: float = 3.0                 # logit boost of a heavy hitter, in std units
    temp_log2_range: tuple[float, float] | None = None   # per-KV-head key temperature 2^U(a,b)
    page_bytes: int = 4096
    prompt_grant_slack: int = 1
    reclaim_in_decode: int = 1
    note: str = ""
    shape: str = ""                          # the model the layer is shaped like

    @property
    def n_q_heads(self) -> int:
        return self.n_kv_heads * self.group_size

    def max_seq_len(self) -> int:
        hi = self.prompt_len if isinstance(self.prompt_len, int) else self.prompt_len[1]
        return hi + self.decode_steps

    def pool_config(self, **over) -> dict:
        cfg = dict(
            n_layers=self.n_layers, n_kv_heads=self.n_kv_heads, group_size=self.group_size,
            head_dim=HEAD_DIM, page_bytes=self.page_bytes, n_pages=self.n_pages,
            max_requests=self.n_requests, max_seq_len=self.max_seq_len(),
            tokens_per_hi_page=0, tokens_per_lo_page=0, lo_enabled=self.lo_enabled,
            alpha_h=self.alpha_h, alpha_l=self.alpha_l, recent_window=self.recent_window,
            obs_window=OBS_WINDOW, prompt_grant_slack=self.prompt_grant_slack,
            reclaim_in_decode=self.reclaim_in_decode)
        cfg.update(over)
        return cfg


# Page size: 4 KB for tiny (its stated configuration); 3.5 KB for the
# model-shaped layers, where the page-fill rule gives 16 hi / 32 lo tokens per
# page (93% / 100% of the page used, against 91% / 98% at 4 KB) and every
# 16-token attention chunk lies inside one page.
WORKLOADS: dict[str, Workload] = {
    # 1 layer, 2 requests (ctx 512 and 700), 2 KV heads x GQA 4, N(0,1) K/V with
    # 4 outlier channels x8, 4 KB pages.
    "tiny": Workload("tiny", n_layers=1, n_kv_heads=2, group_size=4, n_requests=2,
                     prompt_len=(512, 700), decode_steps=64, n_pages=1024,
                     note="prompt lengths are exactly 512 and 700"),
    # Llama-3-8B-shaped layer: 32 q / 8 KV heads, batch 32, ctx 4096, rank-4 bias.
    "llama8b": Workload("llama8b", n_layers=1, n_kv_heads=8, group_size=4, n_requests=32,
                        prompt_len=4096, decode_steps=128, n_pages=84800, bias_rank=4,
                        page_bytes=3584, shape="Llama-3-8B"),
    # Llama-3-70B-shaped layer: 64 q / 8 KV heads, batch 8, ctx 32768, 2% heavy hitters.
    "llama70b": Workload("llama70b", n_layers=1, n_kv_heads=8, group_size=8, n_requests=8,
                         prompt_len=32768, decode_steps=32, n_pages=164096, bias_rank=4,
                         heavy_frac=0.02, page_bytes=3584, shape="Llama-3-70B"),
    # QwQ-32B-shaped long generation: 40 q / 8 KV heads, batch 64, 1024-token prompt,
    # 8192 decode steps with compaction every step and tail-page frees.
    "qwq32b": Workload("qwq32b", n_layers=1, n_kv_heads=8, group_size=5, n_requests=64,
                       prompt_len=1024, decode_steps=8192, n_pages=230000, bias_rank=4,
                       page_bytes=3584, shape="QwQ-32B"),
    # Qwen2.5-7B-shaped GQA-7: 28 q / 4 KV heads, batch 128, ctx U{1K..16K}, lo tier off,
    # skewed per-head sparsity from a per-KV-head key temperature.
    "qwen7b": Workload("qwen7b", n_layers=1, n_kv_heads=4, group_size=7, n_requests=128,
                       prompt_len=(1024, 16384), decode_steps=16, n_pages=350000, page_bytes=3584,
                       lo_enabled=0, temp_log2_range=(0.5, 3.5), shape="Qwen2.5-7B"),
}


# The three-tier variant of a workload (its pool configuration only; the
# inputs are the workload's own): a mid tier K8V2 between hi and lo from
# alpha_m / N = 1 / N, 16 tokens per mid page (the attention kernel's chunk),
# two slack pages in the prompt grant for the three partial pages a head can
# leave.
THREE_TIER = dict(mid_enabled=1, alpha_m=1.0, tokens_per_mid_page=16, prompt_grant_slack=2)


def _rng(name: str, seed: int, role: str, step: int = 0) -> np.random.Generator:
    key = zlib.crc32(f"{name}/{role}".encode())
    return np.random.default_rng([seed, key, step])


def prompt_lengths(w: Workload, seed: int = 0) -> np.ndarray:
    if w.name == "tiny":
        return np.array([512, 700], dtype=np.int32)
    if isinstance(w.prompt_len, int):
        return np.full(w.n_requests, w.prompt_len, dtype=np.int32)
    lo, hi = w.prompt_len
    return _rng(w.name, seed, "lens").integers(lo, hi + 1, size=w.n_requests).astype(np.int32)


def _normal16(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


@dataclass
class HeadStructure:
    """Per-KV-head structure shared by prompt and decode draws."""
    outlier_idx: np.ndarray          # [Hkv, n_outlier] channel indices
    bias_k: np.ndarray | None        # [Hkv, 128, r]
    bias_v: np.ndarray | None        # [Hkv, 128, r]
    q_coef: np.ndarray | None        # [Hq, r] per query head
    temp: np.ndarray | None          # [Hkv] key temperature


def head_structure(w: Workload, seed: int = 0) -> HeadStructure:
    rng = _rng(w.name, seed, "structure")
    hkv = w.n_kv_heads
    idx = np.stack([rng.choice(HEAD_DIM, size=w.outlier_channels, replace=False)
                    for _ in range(hkv)]) if w.outlier_channels else np.zeros((hkv, 0), np.int64)
    bk = bv = qc = None
    if w.bias_rank:
        r = w.bias_rank
        bk = (rng.standard_normal((hkv, HEAD_DIM, r)) * w.bias_std).astype(np.float32)
        bv = (rng.standard_normal((hkv, HEAD_DIM, r)) * w.bias_std).astype(np.float32)
        qc = rng.standard_normal((w.n_q_heads, r)).astype(np.float32)
    temp = None
    if w.temp_log2_range is not None:
        a, b = w.temp_log2_range
        temp = (2.0 ** rng.uniform(a, b, size=hkv)).astype(np.float32)
    return HeadStructure(idx, bk, bv, qc, temp)


def _shape_kv(x: np.ndarray, st: HeadStructure, w: Workload, bias: np.ndarray | None,
              coef: np.ndarray | None) -> np.ndarray:
    """x: [T, Hkv, 128] float32 normals -> structured (in place)."""
    for h in range(w.n_kv_heads):
        if st.outlier_idx.shape[1]:
            x[:, h, st.outlier_idx[h]] *= w.outlier_scale
        if bias is not None and coef is not None:
            x[:, h, :] += coef[:, h, :] @ bias[h].T
    return x


def _shape_q(q: np.ndarray, st: HeadStructure, w: Workload) -> np.ndarray:
    """q: [..., Hq, 128] float32 normals -> plus the head's bias direction."""
    if st.bias_k is not None:
        for hq in range(w.n_q_heads):
            q[..., hq, :] += st.bias_k[hq // w.group_size] @ st.q_coef[hq]
    return q


def prompt_inputs(name: str, seed: int = 0, requests: list[int] | None = None) -> dict:
    """Prompt-phase inputs of a workload.

    Returns k, v: fp16 [sum(lens), Hkv, 128] (requests back to back), q_obs: fp16
    [R, 32, Hq, 128] (row o = position len-32+o), lens: int32 [R]. `requests`
    restricts the draw to a subset of request indices (same values as in the
    full draw, since every request has its own stream)."""
    w = WORKLOADS[name]
    st = head_structure(w, seed)
    lens_all = prompt_lengths(w, seed)
    reqs = list(range(w.n_requests)) if requests is None else list(requests)
    ks, vs, qs = [], [], []
    for r in reqs:
        n = int(lens_all[r])
        rng = _rng(name, seed, "prompt", r)
        k = _normal16(rng, (n, w.n_kv_heads, HEAD_DIM))
        v = _normal16(rng, (n, w.n_kv_heads, HEAD_DIM))
        q = _normal16(rng, (OBS_WINDOW, w.n_q_heads, HEAD_DIM))
        ck = cv = None
        if w.bias_rank:
            ck = rng.standard_normal((n, w.n_kv_heads, w.bias_rank)).astype(np.float32)
            cv = rng.standard_normal((n, w.n_kv_heads, w.bias_rank)).astype(np.float32)
        _shape_kv(k, st, w, st.bias_k, ck)
        _shape_kv(v, st, w, st.bias_v, cv)
        _shape_q(q, st, w)
        if st.temp is not None:
            k *= st.temp[None, :, None]
        if w.heavy_frac > 0:
            _add_heavy_hitters(k, q, w, rng)
        ks.append(k.astype(np.float16))
        vs.append(v.astype(np.float16))
        qs.append(q.astype(np.float16))
    return dict(k=np.concatenate(ks), v=np.concatenate(vs), q_obs=np.stack(qs),
                lens=lens_all[reqs].astype(np.int32))


def prefill_inputs(name: str, seed: int = 0, requests: list[int] | None = None,
                   max_len: int | None = None) -> dict:
    """Inputs of the prompt's own attention: prompt_inputs plus q fp16
    [sum(lens), Hq, 128], every prompt position's query (requests back to
    back). The last 32 rows of each request are its observation queries
    (q_obs row o = position len-32+o); the earlier rows come from a stream of
    their own with the same per-head structure. max_len truncates every
    prompt to its first max_len tokens, whose last 32 rows then form q_obs."""
    w = WORKLOADS[name]
    st = head_structure(w, seed)
    base = prompt_inputs(name, seed, requests)
    reqs = list(range(w.n_requests)) if requests is None else list(requests)
    ks, vs, qs, qo, lens = [], [], [], [], []
    t0 = 0
    for i, r in enumerate(reqs):
        n = int(base["lens"][i])
        rng = _rng(name, seed, "prefill_q", r)
        early = _normal16(rng, (max(n - OBS_WINDOW, 0), w.n_q_heads, HEAD_DIM))
        _shape_q(early, st, w)
        q = np.concatenate([early.astype(np.float16), base["q_obs"][i][max(OBS_WINDOW - n, 0):]])
        m = n if max_len is None else min(n, max_len)
        ks.append(base["k"][t0:t0 + m]); vs.append(base["v"][t0:t0 + m]); qs.append(q[:m])
        obs = np.zeros((OBS_WINDOW, w.n_q_heads, HEAD_DIM), np.float16)
        take = min(m, OBS_WINDOW)
        obs[OBS_WINDOW - take:] = q[m - take:m]
        qo.append(obs)
        lens.append(m)
        t0 += n
    return dict(k=np.concatenate(ks), v=np.concatenate(vs), q=np.concatenate(qs), q_obs=np.stack(qo),
                lens=np.array(lens, dtype=np.int32))


def _add_heavy_hitters(k: np.ndarray, q: np.ndarray, w: Workload, rng: np.random.Generator):
    """Give heavy_frac of the keys outside the recent window a key component
    along the unit mean of the group's observation queries, sized so that the
    mean query's logit rises by heavy_sigma standard deviations of its base
    logits."""
    n = k.shape[0]
    eligible = max(0, n - w.recent_window)
    cnt = int(round(w.heavy_frac * eligible))
    if cnt == 0:
        return
    for h in range(w.n_kv_heads):
        qg = q[:, h * w.group_size:(h + 1) * w.group_size, :].reshape(-1, HEAD_DIM)
        mean_q = qg.mean(axis=0)
        unit = mean_q / np.linalg.norm(mean_q)
        base = (k[:, h, :] @ mean_q) / np.sqrt(HEAD_DIM)
        sigma = float(base.std())
        delta = w.heavy_sigma * sigma * np.sqrt(HEAD_DIM) / float(np.linalg.norm(mean_q))
        pos = rng.choice(eligible, size=cnt, replace=False)
        k[pos, h, :] += delta * unit


def decode_inputs(name: str, step: int, seed: int = 0, requests: list[int] | None = None) -> dict:
    """Inputs of decode step `step`: new k, v fp16 [R, Hkv, 128] and query q fp16
    [R, Hq, 128], with the same per-head structure as the prompt."""
    w = WORKLOADS[name]
    st = head_structure(w, seed)
    reqs = list(range(w.n_requests)) if requests is None else list(requests)
    rng = _rng(name, seed, "decode", step)
    r_all = w.n_requests
    k = _normal16(rng, (r_all, w.n_kv_heads, HEAD_DIM))
    v = _normal16(rng, (r_all, w.n_kv_heads, HEAD_DIM))
    q = _normal16(rng, (r_all, w.n_q_heads, HEAD_DIM))
    if w.bias_rank:
        ck = rng.standard_normal((r_all, w.n_kv_heads, w.bias_rank)).astype(np.float32)
        cv = rng.standard_normal((r_all, w.n_kv_heads, w.bias_rank)).astype(np.float32)
        _shape_kv(k, st, w, st.bias_k, ck)
        _shape_kv(v, st, w, st.bias_v, cv)
    else:
        _shape_kv(k, st, w, None, None)
        _shape_kv(v, st, w, None, None)
    _shape_q(q, st, w)
    if st.temp is not None:
        k *= st.temp[None, :, None]
    return dict(k=k[reqs].astype(np.float16), v=v[reqs].astype(np.float16),
                q=q[reqs].astype(np.float16))


def given_scores(n_tokens: int, n_kv_heads: int, seed: int, scale: float = 1.0,
                 zero_frac: float = 0.05) -> np.ndarray:
    """Caller-given token scores (fp32 [n_tokens, Hkv]) for tests that feed the
    compaction path scores directly: log-uniform over ~6 decades with a
    fraction of exact zeros, times `scale`."""
    rng = np.random.default_rng([seed, 0x5C0E])
    s = 10.0 ** rng.uniform(-5.0, 1.0, size=(n_tokens, n_kv_heads))
    s[rng.random((n_tokens, n_kv_heads)) < zero_frac] = 0.0
    return (s * scale).astype(np.float32)


def random_fp16(shape, seed: int, scale: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng([seed, 0xF16])
    return (rng.standard_normal(shape, dtype=np.float32) * scale).astype(np.float16)


def describe(name: str) -> dict:
    d = asdict(WORKLOADS[name])
    d["n_q_heads"] = WORKLOADS[name].n_q_heads
    return d

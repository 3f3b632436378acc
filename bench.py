#!/usr/bin/env python
"""Benchmark of the differentiated-KV hot path on GB300 (one process per GPU).

One step = one pass of the whole path over one batch of the Llama-3-8B-shaped
workload (32 requests x 4096-token prompts, 32 q / 8 KV heads):
  prompt compact_step (score, classify, grant, pack, reclaim)
  then 128 decode steps: [L2 flush] decode compact_step + decode_attention
  (with score update), then free_request for every request.
value = decode-attention GB/s: algorithmic bytes (hi token 200 B, lo token
104 B, +8 B score update, + q and out) over the device time of one
decode_attention call timed alone between CUDA events on its stream (L2
flushed before each decode step). compact_step is reported in us per layer.

The same loop then runs, untimed for the headline, on the 70B-shaped layer,
on the 8B-shaped layer with 4 KB pages (the kernel for any page geometry),
and on the Qwen2.5-7B-shaped GQA-7 batch; their figures, each with its own
fraction of the HBM roofline, are in `parts`. `parts.prefill` times the
prompt's own causal attention (TFLOP/s against the tensor-core roofline) and
the prompt compact_step that takes that attention's log-sum-exps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dkv|reference]

With --gpus N > 1 outside torchrun the script starts N ranks itself (one
process per GPU, torch.distributed.run on 127.0.0.1).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import tempfile
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "compressed-KV decode attn GB/s (% of GB300 HBM peak); compact_step µs/layer"
HI_BYTES, LO_BYTES, SCORE_RMW = 200, 104, 8
MID_BYTES = 168          # the three-tier variant's mid token: 8-bit key, 2-bit value, metadata
# kernels the library launches: prompt compact_step (setup, two tensor-core
# scoring passes, lse merge, classification, three plan kernels, scatter,
# pack), decode compact_step (plan, alloc, apply), decode attention
# (attention, epilogue), free_request (one)
LAUNCHES = {"prompt": 10, "decode": 3, "attention": 2, "free": 1}

# DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum, caches
# flushed by ncu before each kernel) of the llama8b bench step:
#   one decode-attention call (k_attn_paged + k_attn_epi, third decode step);
#   one prompt compact_step (its 10 kernels, timed step).
# Valid only for the kernel sources they were taken on: any change to them
# makes the bench report null until a new capture replaces the record.
ATTN_TRAFFIC = {
    "workload": "llama8b",
    "bytes_per_call": 114_553_600 + 2_715_648 + 26_332_928,
    "sources": {
        "attention.cu": "4787725370c06619bafc550a320ea946f0b37b4ab4c2c0246628090ae0b54317",
        "dkv_common.cuh": "ba5510123ecbe1069424c0470463527dccb53b0444f61c6e606f7028ef848f8c",
        "dkv_kernels.cuh": "ec4d6d05af74cad9f54d34cff8dd36f8a38b036a2e5483df855c71eea66bd45b",
    },
}
PROMPT_TRAFFIC = {
    "workload": "llama8b",
    "bytes_per_call": 1_018_318_592 + 103_008_000,
    "sources": {
        "prompt.cu": "112318ce1a431d52729ded02427ab6e7b9e88199071cb46c7cfdd9ec55d07845",
        "prompt_tc.cu": "fa63d0ced7a2f9d8266fe4673083378e67dddf037238d1f050656313a455b8c1",
        "alloc.cu": "3cb94c20d08da98fe7db21a35c9243c2b56696d18fe5239f842f1bd8ca6b512a",
        "dkv_tc.cuh": "acb3452effe630c9cbc898bc8a87929dbf4ecd2f43abeb537319b63ad151c2fb",
        "dkv_common.cuh": "ba5510123ecbe1069424c0470463527dccb53b0444f61c6e606f7028ef848f8c",
        "dkv_kernels.cuh": "ec4d6d05af74cad9f54d34cff8dd36f8a38b036a2e5483df855c71eea66bd45b",
    },
}
L2_FLUSH_BYTES = 256 << 20


def recorded_traffic(record: dict, workload: str, page_bytes: int | None = None):
    """A recorded DRAM-traffic figure when the kernel sources still hash to
    those it was captured on (and the workload is the one captured), else None."""
    if workload != record["workload"] or page_bytes not in (None, workloads.WORKLOADS[workload].page_bytes):
        return None
    csrc = os.path.join(ROOT, "differentiated_kv_cache_gb300", "csrc")
    for name, digest in record["sources"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return record["bytes_per_call"]


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


def hbm_peak():
    p = peaks()
    if "hbm_gbs" in p:
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense fp16/bf16 tensor-core peak for a kernel timed alone (burst)."""
    p = peaks()
    if "bf16_tflops" in p:
        return float(p["bf16_tflops"]), "measured bf16 burst"
    return 1900.0, "fallback"


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"dkv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self) -> dict:
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend)
    return dist


def reduce_max(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(n: int) -> int:
    """Run this script as n ranks on this node (one process per GPU) and
    return the launcher's exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


# --------------------------------------------------------------- workload
def attn_bytes(hi_tokens: int, lo_tokens: int, n_req: int, hq: int, update: bool, mid_tokens: int = 0) -> int:
    per = HI_BYTES * hi_tokens + LO_BYTES * lo_tokens + MID_BYTES * mid_tokens
    if update:
        per += SCORE_RMW * (hi_tokens + lo_tokens + mid_tokens)
    return per + n_req * hq * (128 * 2 + 128 * 4)


def prompt_bytes(hi_tokens: int, lo_tokens: int, n_tokens_heads: int, n_req: int, hq: int,
                 mid_tokens: int = 0) -> int:
    return 512 * n_tokens_heads + 208 * hi_tokens + 112 * lo_tokens + 176 * mid_tokens + n_req * 32 * hq * 256


def describe(w, lens, T, page_bytes, mid: bool = False) -> str:
    rng = f"{min(lens)}" if min(lens) == max(lens) else f"U{{{min(lens)}..{max(lens)}}}"
    return (f"{w.name}: {w.shape or 'synthetic'}-shaped layer, {len(lens)} requests x {rng}-token prompts, "
            f"{w.n_q_heads} q / {w.n_kv_heads} KV heads, d=128, {page_bytes}-byte pages, "
            f"{T} decode steps with compaction and score update" + ("" if w.lo_enabled else ", low tier off") +
            (", three tiers (hi K8V4 above 2/N, mid K8V2 from 1/N, lo K4V2 from 0.25/N)" if mid else ""))


class Loop:
    """One workload on one GPU: its pool, device-resident inputs and the
    benchmark step (prompt, T x [flush, decode compaction, attention with
    score update], free every request)."""

    def __init__(self, dkv, name: str, seed: int, dev, decode_steps: int | None = None,
                 page_bytes: int | None = None, inputs=None, pool_over: dict | None = None):
        import torch
        self.dkv, self.torch, self.dev = dkv, torch, dev
        self.w = w = workloads.WORKLOADS[name]
        self.T = w.decode_steps if decode_steps is None else decode_steps
        self.inp = inputs if inputs is not None else workloads.prompt_inputs(name, seed)
        self.dec = [workloads.decode_inputs(name, t, seed) for t in range(self.T)]
        self.lens = [int(x) for x in self.inp["lens"]]
        cfg = w.pool_config()
        cfg["max_seq_len"] = max(self.lens) + self.T
        if page_bytes:
            cfg["page_bytes"] = page_bytes
        cfg.update(pool_over or {})
        self.mid = bool(cfg.get("mid_enabled", 0))
        self.page_bytes = cfg["page_bytes"]
        self.cfg = cfg
        self.pool = dkv.dkv_pool_create(dkv.make_config(**{k: v for k, v in cfg.items()
                                                          if k in dict(dkv.dkv_config._fields_)}), dev.index)
        self.slots = list(range(w.n_requests))
        self.k_d = torch.from_numpy(self.inp["k"]).to(dev)
        self.v_d = torch.from_numpy(self.inp["v"]).to(dev)
        self.q_d = torch.from_numpy(self.inp["q_obs"]).to(dev)
        self.dk = torch.from_numpy(np.stack([d["k"] for d in self.dec])).to(dev)
        self.dv = torch.from_numpy(np.stack([d["v"] for d in self.dec])).to(dev)
        self.dq = torch.from_numpy(np.stack([d["q"] for d in self.dec])).to(dev)
        self.out = torch.zeros((w.n_requests, w.n_q_heads, 128), dtype=torch.float32, device=dev)
        # L2 flush between decode steps: write a buffer larger than L2, then
        # read a second one so that the write-back of the dirty lines happens
        # here and not inside the next timed kernel; L2 then holds none of the
        # path's data.
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()

    def close(self):
        self.dkv.dkv_pool_destroy(self.pool)
        self.pool = None

    def launches_per_step(self) -> int:
        return LAUNCHES["prompt"] + self.T * (LAUNCHES["decode"] + LAUNCHES["attention"]) + \
            len(self.slots) * LAUNCHES["free"]

    def step(self, record=None, counts=None):
        """One pass of the path. record: dict of event-pair lists; counts:
        list to fill with (phase, hi, lo) stored tokens (syncs)."""
        dkv, torch, st = self.dkv, self.torch, self.stream
        ev = lambda: torch.cuda.Event(enable_timing=True)
        if record is not None:
            e0, e1 = ev(), ev()
            e0.record(st)
        dkv.dkv_compact_step(self.pool, 0, dkv.DKV_PROMPT, self.slots, self.lens, self.k_d, self.v_d, self.q_d)
        if record is not None:
            e1.record(st)
            record["prompt"].append((e0, e1))
        if counts is not None:
            s = dkv.dkv_pool_status(self.pool)
            counts.append(("prompt", s["hi_tokens"], s["lo_tokens"], s["mid_tokens"]))
        for t in range(self.T):
            self.flush.fill_(t & 0xFF)
            torch.amax(self.flush_rd)
            # Even steps put an event between compaction and attention: the
            # compaction and the call are timed alone. Odd steps do not: there
            # the attention kernel launches while the compaction drains, as in
            # a decode loop, and (compaction + attention) is timed as one.
            split = t % 2 == 0
            if record is not None:
                c0, c1, a1 = ev(), ev(), ev()
                c0.record(st)
            dkv.dkv_compact_step(self.pool, 0, dkv.DKV_DECODE, self.slots, None, self.dk[t], self.dv[t])
            if record is not None and split:
                c1.record(st)
            dkv.dkv_decode_attention(self.pool, 0, self.slots, self.dq[t], self.out, True)
            if record is not None:
                a1.record(st)
                if split:
                    record["compact"].append((c0, c1))
                    record["attn_alone"].append((c1, a1))
                else:
                    record["pair"].append((c0, a1))
            if counts is not None:
                s = dkv.dkv_pool_status(self.pool)
                counts.append(("attn", s["hi_tokens"], s["lo_tokens"], s["mid_tokens"]))
        for s in self.slots:
            dkv.dkv_free_request(self.pool, s)

    def warm(self, n: int):
        counts = []
        for i in range(max(n, 1)):
            self.step(counts=counts if i == 0 else None)
        self.torch.cuda.synchronize()
        st = self.dkv.dkv_pool_status(self.pool)
        assert st["error"] == 0, st
        self.prompt_counts = counts[0]
        w = self.w
        self.bytes_per_attn = [attn_bytes(c[1], c[2], w.n_requests, w.n_q_heads, True, c[3])
                               for c in counts if c[0] == "attn"]
        self.n_th = sum(self.lens) * w.n_kv_heads
        self.pbytes = prompt_bytes(self.prompt_counts[1], self.prompt_counts[2], self.n_th, w.n_requests,
                                   w.n_q_heads, self.prompt_counts[3])

    def timed(self, steps: int) -> dict:
        torch = self.torch
        rec = {"prompt": [], "compact": [], "attn_alone": [], "pair": []}
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        for _ in range(steps):
            self.step(record=rec)
        t1.record(self.stream)
        torch.cuda.synchronize()
        ms = lambda pairs: [a.elapsed_time(b) for a, b in pairs]
        r = {"step_ms": t0.elapsed_time(t1) / steps, "prompt_ms": statistics.mean(ms(rec["prompt"])),
             "compact_ms": statistics.mean(ms(rec["compact"])),
             "alone_ms": statistics.mean(ms(rec["attn_alone"]))}
        # in the loop: (compaction + attention) of the odd steps less the
        # compaction alone of the even steps
        r["pair_ms"] = statistics.mean(ms(rec["pair"])) if rec["pair"] else r["compact_ms"] + r["alone_ms"]
        r["loop_ms"] = r["pair_ms"] - r["compact_ms"] if rec["pair"] else r["alone_ms"]
        r["attn_bytes"] = sum(self.bytes_per_attn) / len(self.bytes_per_attn)
        return r

    def summary(self, r: dict, peak: float) -> dict:
        """Per-workload figures, each against the HBM roofline."""
        gbs = lambda b, ms: b / (ms * 1e-3) / 1e9
        a_alone, a_loop = gbs(r["attn_bytes"], r["alone_ms"]), gbs(r["attn_bytes"], r["loop_ms"])
        p = gbs(self.pbytes, r["prompt_ms"])
        pc = self.prompt_counts
        return {
            "workload": describe(self.w, self.lens, self.T, self.page_bytes, self.mid),
            "decode_attention_us": round(r["alone_ms"] * 1e3, 2),
            "decode_attention_gbs": round(a_alone, 1), "decode_attention_frac": round(a_alone / peak, 4),
            "decode_attention_in_loop_us": round(r["loop_ms"] * 1e3, 2),
            "decode_attention_in_loop_gbs": round(a_loop, 1),
            "decode_attention_in_loop_frac": round(a_loop / peak, 4),
            "attention_bytes_per_call": int(r["attn_bytes"]),
            "compact_step_prompt_us_per_layer": round(r["prompt_ms"] * 1e3, 1),
            "compact_step_prompt_gbs": round(p, 1), "compact_step_prompt_frac": round(p / peak, 4),
            "compact_step_prompt_bytes": int(self.pbytes),
            "compact_step_decode_us_per_layer": round(r["compact_ms"] * 1e3, 2),
            # one generation step of the decode loop: compaction and the
            # attention call with score update, timed as one (odd steps)
            "generation_step_us": round(r["pair_ms"] * 1e3, 2),
            "stored_tokens_after_prompt": {"hi": pc[1], "lo": pc[2], "pruned": self.n_th - pc[1] - pc[2] - pc[3],
                                           **({"mid": pc[3]} if self.mid else {})},
            "kv_bytes_vs_fp16": round((HI_BYTES * pc[1] + LO_BYTES * pc[2] + MID_BYTES * pc[3]) / (self.n_th * 512),
                                      4),
        }


# ------------------------------------------------------------------ churn
def run_churn(dkv, dev, seed: int, ticks: int, peak: float) -> dict:
    """QwQ-32B-shaped long generation with requests arriving and finishing
    (40 q / 8 KV heads, 1024-token prompts, U{128..512} generated tokens, at
    most 64 at once): every tick admits waiting requests whose grant and
    growth fit (one prompt compact_step), runs one generation compact_step
    and one decode_attention with score update over every active request, and
    frees the finished ones, so that the free list's counters wrap the pool.
    Compaction and attention are timed alone with CUDA events."""
    import torch
    name = "qwq32b"
    w = workloads.WORKLOADS[name]
    H, Hq, R = w.n_kv_heads, w.n_q_heads, w.n_requests
    gen_lo, gen_hi, n0 = 128, 512, 1024
    n_pages = 32000
    cfg = w.pool_config(n_pages=n_pages, max_seq_len=n0 + gen_hi + 1)
    pool = dkv.dkv_pool_create(dkv.make_config(**{k: v for k, v in cfg.items()
                                                  if k in dict(dkv.dkv_config._fields_)}), dev.index)
    t_hi = dkv.dkv_pool_geometry(pool)["t_hi"]
    rng = np.random.default_rng([seed, 0xC4])
    inp = workloads.prompt_inputs(name, seed, requests=list(range(8)))
    pk = torch.from_numpy(inp["k"]).to(dev)
    pv_ = torch.from_numpy(inp["v"]).to(dev)
    pq = torch.from_numpy(inp["q_obs"]).to(dev)
    steps = [workloads.decode_inputs(name, t, seed) for t in range(16)]
    dk = [torch.from_numpy(d["k"]).to(dev) for d in steps]
    dv = [torch.from_numpy(d["v"]).to(dev) for d in steps]
    dq = [torch.from_numpy(d["q"]).to(dev) for d in steps]
    out = torch.empty((R, Hq, 128), dtype=torch.float32, device=dev)
    st_ = torch.cuda.current_stream()
    active, done = {}, 0
    growth = lambda g: 2 * H * (g // t_hi + 2)
    grant = H * (-(-n0 // t_hi) + 1)
    comp, att, nact, abytes = [], [], [], []
    ev = lambda: torch.cuda.Event(enable_timing=True)
    for tick in range(ticks):
        s = dkv.dkv_pool_status(pool)
        assert s["error"] == 0, s
        budget = s["free_pages"] - sum(growth(t - g) for g, t in active.values())
        new = []
        for slot in range(R):
            if slot in active or budget < grant + growth(gen_hi):
                continue
            active[slot] = [0, int(rng.integers(gen_lo, gen_hi + 1))]
            budget -= grant + growth(active[slot][1])
            new.append(slot)
        for j in range(0, len(new), 8):      # prompts of 8 requests (the drawn inputs' batch)
            sl = new[j:j + 8]
            r = len(sl)
            dkv.dkv_compact_step(pool, 0, dkv.DKV_PROMPT, sl, [n0] * r, pk[:r * n0], pv_[:r * n0], pq[:r])
        if not active:
            continue
        slots = sorted(active)
        n = len(slots)
        x = tick % len(steps)
        # the status read above left the GPU idle: a short device wait lets the
        # tick's launches queue up behind it, so the events time the kernels
        # and not the host's launch calls
        torch.cuda._sleep(200_000)
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(st_)
        dkv.dkv_compact_step(pool, 0, dkv.DKV_DECODE, slots, None, dk[x][:n], dv[x][:n])
        e1.record(st_)
        dkv.dkv_decode_attention(pool, 0, slots, dq[x][:n], out[:n], True)
        e2.record(st_)
        comp.append((e0, e1))
        att.append((e1, e2))
        nact.append(n)
        abytes.append(attn_bytes(s["hi_tokens"], s["lo_tokens"], n, Hq, True))
        for slot in slots:
            active[slot][0] += 1
            if active[slot][0] >= active[slot][1]:
                dkv.dkv_free_request(pool, slot)
                del active[slot]
                done += 1
    torch.cuda.synchronize()
    s = dkv.dkv_pool_status(pool)
    assert s["error"] == 0, s
    dkv.dkv_pool_destroy(pool)
    c_us = [a.elapsed_time(b) * 1e3 for a, b in comp][16:]
    a_us = [a.elapsed_time(b) * 1e3 for a, b in att][16:]
    gbs = sum(abytes[16:]) / (sum(a_us) * 1e-6) / 1e9
    return {"workload": f"{name}: QwQ-32B-shaped layer, {Hq} q / {H} KV heads, {n0}-token prompts, "
                        f"U{{{gen_lo}..{gen_hi}}} generated tokens each, at most {R} requests at once, "
                        f"{n_pages} pages, {ticks} ticks of admit / compact / attend / free",
            "requests_finished": done, "mean_active": round(float(np.mean(nact)), 1),
            "compact_step_decode_us_per_layer": round(float(np.mean(c_us)), 2),
            "decode_attention_us": round(float(np.mean(a_us)), 2), "decode_attention_gbs": round(gbs, 1),
            "decode_attention_frac": round(gbs / peak, 4),
            "list_start": s["list_start"], "list_end": s["list_end"], "list_wraps": s["list_end"] // n_pages}


# ---------------------------------------------------------------- prefill
def prefill_flops(lens, hq: int) -> float:
    """Algorithmic FLOPs of causal attention over the prompts: q.k and p.v,
    2 d each, for every (query, key <= query) pair of every query head."""
    return float(sum(4 * 128 * n * (n + 1) // 2 for n in lens) * hq)


def run_prefill(dkv, dev, name: str, seed: int, reps: int, peak: float, n_req: int | None = None) -> dict:
    """The prompt's own causal attention (dkv_prefill_attention) and the
    PROMPT compaction that takes its observation rows' log-sum-exps
    (dkv_compact_step_prefilled) beside the compaction that computes them
    itself (dkv_compact_step), each timed alone with CUDA events from a
    flushed L2 on the same batch."""
    import torch
    w = workloads.WORKLOADS[name]
    inp = workloads.prefill_inputs(name, seed, None if n_req is None else list(range(n_req)))
    lens = [int(x) for x in inp["lens"]]
    Hq = w.n_q_heads
    cfg = w.pool_config()
    pool = dkv.dkv_pool_create(dkv.make_config(**{k: v for k, v in cfg.items()
                                                  if k in dict(dkv.dkv_config._fields_)}), dev.index)
    q = torch.from_numpy(inp["q"]).to(dev)
    k = torch.from_numpy(inp["k"]).to(dev)
    v = torch.from_numpy(inp["v"]).to(dev)
    qo = torch.from_numpy(inp["q_obs"]).to(dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((len(lens), Hq, 32), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    st_ = torch.cuda.current_stream()
    slots = list(range(len(lens)))
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn, after=None):
        ts = []
        for it in range(reps + 2):
            flush.fill_(it & 0xFF)
            torch.amax(flush_rd)
            torch.cuda._sleep(200_000)      # the launches queue behind a device wait
            e0, e1 = ev(), ev()
            e0.record(st_)
            fn()
            e1.record(st_)
            if after is not None:
                after()
            if it >= 2:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ts)

    def free_all():
        for s_ in slots:
            dkv.dkv_free_request(pool, s_)

    pf_ms = timed(lambda: dkv.dkv_prefill_attention(pool, lens, q, k, v, out, lse))
    cp_ms = timed(lambda: dkv.dkv_compact_step_prefilled(pool, 0, slots, lens, k, v, qo, lse), free_all)
    dkv.dkv_compact_step_prefilled(pool, 0, slots, lens, k, v, qo, lse)
    s = dkv.dkv_pool_status(pool)
    assert s["error"] == 0, s
    counts = (s["hi_tokens"], s["lo_tokens"])
    free_all()
    cs_ms = timed(lambda: dkv.dkv_compact_step(pool, 0, dkv.DKV_PROMPT, slots, lens, k, v, qo), free_all)
    s = dkv.dkv_pool_status(pool)
    assert s["error"] == 0, s
    dkv.dkv_pool_destroy(pool)
    n_th = sum(lens) * w.n_kv_heads
    pbytes = prompt_bytes(counts[0], counts[1], n_th, len(lens), Hq)
    fl = prefill_flops(lens, Hq)
    tf = fl / (pf_ms * 1e-3) / 1e12
    tpk, tkind = tensor_peak()
    gb = lambda ms: pbytes / (ms * 1e-3) / 1e9
    return {
        "workload": f"{name}: {w.shape}-shaped layer, {len(lens)} prompts of {lens[0]} tokens, {Hq} q / "
                    f"{w.n_kv_heads} KV heads, d=128, fp16 q/k/v, fp32 out",
        "prefill_attention_ms": round(pf_ms, 3),
        "prefill_attention_tflops": round(tf, 1),
        "prefill_attention_frac": round(tf / tpk, 4),
        "prefill_peak": f"{tpk} TFLOP/s ({tkind}; fp16 and bf16 share the tensor-core rate)",
        "prefill_flops": fl,
        "prefill_flops_are": "algorithmic: 4 d per causal (query, key) pair per query head; the kernel "
                             "executes 1.5x (the probabilities enter the value product as an fp16 pair)",
        "compact_step_prefilled_us_per_layer": round(cp_ms * 1e3, 1),
        "compact_step_prefilled_gbs": round(gb(cp_ms), 1),
        "compact_step_prefilled_frac": round(gb(cp_ms) / peak, 4),
        "compact_step_same_batch_us_per_layer": round(cs_ms * 1e3, 1),
        "compact_step_bytes": int(pbytes),
    }


# ------------------------------------------------------------- dkv (GPU)
def run_dkv(args, world, rank, local):
    import torch
    import differentiated_kv_cache_gb300 as dkv
    dkv.build.build()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    peak, peak_kind = hbm_peak()
    # each rank serves its own shard of requests: its own seed, its own pool
    loop = Loop(dkv, args.workload, args.seed + rank, dev, decode_steps=args.decode_steps)
    w = loop.w
    loop.warm(args.warmup)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        r = loop.timed(args.steps)
    barrier(dist)
    step_ms_max = reduce_max(dist, r["step_ms"], dev)
    call_ms_max = reduce_max(dist, r["alone_ms"], dev)
    all_bytes = reduce_sum(dist, r["attn_bytes"], dev)
    value = all_bytes / (call_ms_max * 1e-3) / 1e9
    achieved = r["attn_bytes"] / (r["alone_ms"] * 1e-3) / 1e9
    parts = loop.summary(r, peak)
    parts["compact_step_prompt_traffic"] = recorded_traffic(PROMPT_TRAFFIC, args.workload)
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic (seeded numpy; model-shaped K/V/Q, no weights or datasets)",
        "config": {
            "workload": parts["workload"],
            "requests": w.n_requests, "prompt_len": loop.lens[0], "decode_steps": loop.T,
            "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "alpha_h": w.alpha_h, "alpha_l": w.alpha_l,
            "window": w.recent_window, "page_bytes": loop.page_bytes,
            "l2": "flushed before every decode step, outside the timed events: 256 MiB written, then a "
                  "second 256 MiB read (L2 left clean); prompt inputs 537 MB > L2",
            "value_is": "decode-attention algorithmic bytes / device time of one decode_attention call timed "
                        "alone between CUDA events on its stream (even decode steps), max over ranks; "
                        "parts.decode_attention_in_loop_* time the call inside the decode loop, where it "
                        "launches while the compaction drains",
            "parallelism": f"{world} independent pools (one per GPU, each its own request shard), "
                           f"no collective in the path",
        },
        "parts": parts,
        "roofline": {"bound": "hbm", "kernel": "dkv_decode_attention call (k_attn_paged + k_attn_epi)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": int(r["attn_bytes"]),
                     "traffic": args.traffic if args.traffic is not None else
                     recorded_traffic(ATTN_TRAFFIC, args.workload)},
        "gpu_launches": args.steps * loop.launches_per_step(),
    }
    result["clocks"] = clk.summary()
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, loop, dist)
    loop.close()
    headline_inputs = loop.inp
    del loop
    torch.cuda.empty_cache()
    # the other configurations, each its own pool, outside the headline's timed region
    extras = [] if args.extras in ("", "none") else args.extras.split(",")
    result["parts"]["other_configs"] = {}
    for name in extras:
        # "<workload>[@<page bytes>][+mid]": +mid runs the workload's inputs on a three-tier pool
        wl, _, pb = name.partition("@")
        three = name.endswith("+mid")
        wl, pb = wl.removesuffix("+mid"), pb.removesuffix("+mid")
        ex = Loop(dkv, wl, args.seed + rank, dev, page_bytes=int(pb) if pb else None,
                  decode_steps=min(workloads.WORKLOADS[wl].decode_steps, 32),
                  inputs=headline_inputs if wl == args.workload else None,
                  pool_over=workloads.THREE_TIER if three else None)
        ex.warm(1)
        rr = ex.timed(args.extra_steps)
        result["parts"]["other_configs"][name] = ex.summary(rr, peak)
        ex.close()
        del ex
        torch.cuda.empty_cache()
    if args.prefill_reps > 0:
        result["parts"]["prefill"] = run_prefill(dkv, dev, args.workload, args.seed + rank, args.prefill_reps,
                                                 peak, args.prefill_requests)
        torch.cuda.empty_cache()
    if args.churn_ticks > 0:
        result["parts"]["churn"] = run_churn(dkv, dev, args.seed + rank, args.churn_ticks, peak)
        torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, loop: Loop, dist):
    """The same step through the C ABI with inputs in pinned host memory:
    every step copies its inputs (the prompt K/V/Q and every decode step's
    K/V/q, staged back to back in one pinned buffer) to the device with one
    copy, runs the path, and reads every decode step's attention output back
    with one copy."""
    import torch
    dkv, dev, w = loop.dkv, loop.dev, loop.w
    T, pool, slots = loop.T, loop.pool, loop.slots
    R, Hq = w.n_requests, w.n_q_heads
    parts = [loop.inp["k"], loop.inp["v"], loop.inp["q_obs"]]
    for d in loop.dec:
        parts += [d["k"], d["v"], d["q"]]
    sizes = [a.size for a in parts]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    hin = torch.empty(int(offs[-1]), dtype=torch.float16).pin_memory()
    hin_np = hin.numpy()
    for a, o in zip(parts, offs[:-1]):
        hin_np[o:o + a.size] = a.reshape(-1)
    din = torch.empty(hin.shape, dtype=torch.float16, device=dev)
    views = [din[int(o):int(o) + a.size].view(a.shape) for a, o in zip(parts, offs[:-1])]
    k_d, v_d, q_d = views[:3]
    dec = [views[3 + 3 * t: 6 + 3 * t] for t in range(T)]
    out = torch.empty((T, R, Hq, 128), dtype=torch.float32, device=dev)
    hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    st = torch.cuda.current_stream()
    slots_np = np.asarray(slots, dtype=np.int32)
    lens_np = np.asarray(loop.lens, dtype=np.int32)

    def step():
        din.copy_(hin, non_blocking=True)
        dkv.dkv_compact_step(pool, 0, dkv.DKV_PROMPT, slots_np, lens_np, k_d, v_d, q_d, stream=st)
        for t in range(T):
            dk, dv, dq = dec[t]
            dkv.dkv_compact_step(pool, 0, dkv.DKV_DECODE, slots_np, None, dk, dv, stream=st)
            dkv.dkv_decode_attention(pool, 0, slots_np, dq, out[t], True, stream=st)
        hout.copy_(out, non_blocking=True)
        for s_ in slots:
            dkv.dkv_free_request(pool, s_, stream=st)
        torch.cuda.synchronize()

    step()
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    dt = reduce_max(dist, dt, dev)
    n = dist.get_world_size() if dist is not None else 1
    attn_bytes_step = sum(loop.bytes_per_attn)
    h2d = int(hin.numel()) * 2
    d2h = int(hout.numel()) * 4
    return {"value": round(n * attn_bytes_step / dt / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(dt * 1e3, 2),
            "what": "decode-attention algorithmic bytes of a step / wall time of the whole step through the "
                    "C ABI: one copy of the step's inputs from pinned host memory (prompt K/V/Q and every "
                    "decode step's K/V/q), the path, one copy of every decode step's output back (host sync "
                    "at the end of each step)"}


# --------------------------------------------------- oracle (CPU baseline)
def _oracle_request(name: str, seed: int, r: int, n_decode: int):
    """The oracle's pool for request r of the workload after its prompt
    compaction (fp64 scoring); returns (pool, prompt seconds)."""
    import oracle
    w = workloads.WORKLOADS[name]
    inp = workloads.prompt_inputs(name, seed, requests=[r])
    n0 = int(inp["lens"][0])
    cfg = w.pool_config(max_requests=1, max_seq_len=n0 + n_decode,
                        n_pages=2 * w.n_kv_heads * (n0 // 16 + n_decode + 8))
    pool = oracle.Pool(cfg)
    t0 = time.perf_counter()
    assert pool.prompt(0, [0], inp["lens"], inp["k"], inp["v"], inp["q_obs"]) == 0
    return pool, time.perf_counter() - t0


def oracle_sample(name: str, seed: int, requests: list[int], n_decode: int, threads: int) -> dict:
    """The oracle as it stands on a bounded sample of the workload: the
    prompt compaction (fp64 scoring) of each sampled request, then n_decode
    decode steps (compaction, then fp64 attention with score update), the
    requests run side by side on `threads` host threads (the oracle's C code
    runs without the GIL; every request has a pool of its own). Times are
    wall-clock over all threads: the prompt phase, and the attention calls
    (decode compaction untimed)."""
    import oracle
    oracle.build()
    w = workloads.WORKLOADS[name]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        res = list(ex.map(lambda r: _oracle_request(name, seed, r, n_decode), requests))
        t_prompt = time.perf_counter() - t0        # includes drawing the inputs
        pools = [p for p, _ in res]
        prompt_cpu = sum(t for _, t in res)
        ab, at = 0, 0.0
        for t in range(n_decode):
            d = [workloads.decode_inputs(name, t, seed, requests=[r]) for r in requests]
            list(ex.map(lambda x: pools[x].decode(0, [0], d[x]["k"], d[x]["v"]), range(len(pools))))
            for p in pools:
                hc = p.head_counts[0, 0]
                ab += attn_bytes(int(hc[:, 0].sum()), int(hc[:, 1].sum()), 1, w.n_q_heads, True)
            t1 = time.perf_counter()
            rcs = list(ex.map(lambda x: pools[x].attention(0, [0], d[x]["q"], update_scores=True)[0],
                              range(len(pools))))
            at += time.perf_counter() - t1
            assert all(rc == 0 for rc in rcs)
    return {"attn_bytes": ab, "attn_s": at, "prompt_wall_s": t_prompt, "prompt_cpu_s": prompt_cpu}


def cpu_baseline(args) -> dict:
    n_dec = 8
    cores = os.cpu_count() or 1
    w = workloads.WORKLOADS[args.workload]
    reqs = list(range(min(cores, w.n_requests)))
    mt = oracle_sample(args.workload, args.seed, reqs, n_dec, threads=len(reqs))
    st = oracle_sample(args.workload, args.seed, [0], n_dec, threads=1)
    return {"value": round(mt["attn_bytes"] / mt["attn_s"] / 1e9, 4), "unit": "GB/s", "cores": len(reqs),
            "kind": "oracle",
            "sample": f"{len(reqs)} of {w.n_requests} requests, one per host thread ({cores} cores seen), "
                      f"{n_dec} decode steps each: decode attention (fp64) timed wall-clock over all threads",
            "value_1thread": round(st["attn_bytes"] / st["attn_s"] / 1e9, 4),
            "compact_step_prompt_us_per_request_layer_1thread": round(st["prompt_cpu_s"] * 1e6, 0),
            "compact_step_prompt_us_per_request_layer": round(mt["prompt_cpu_s"] / len(reqs) * 1e6, 0)}


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    n_dec = 4
    cores = os.cpu_count() or 1
    w = workloads.WORKLOADS[args.workload]
    reqs = list(range(min(cores, w.n_requests)))
    for _ in range(args.warmup):
        oracle_sample(args.workload, args.seed, reqs[:1], 1, threads=1)
    tot_b, tot_t = 0, 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s = oracle_sample(args.workload, args.seed, reqs, n_dec, threads=len(reqs))
        tot_b += s["attn_bytes"]
        tot_t += s["attn_s"]
    t_all = time.perf_counter() - t0
    value = tot_b / tot_t / 1e9
    sample = (f"{len(reqs)} of {w.n_requests} requests, one per host thread, {n_dec} decode steps per step; "
              f"decode attention (fp64) timed wall-clock over all threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_all / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.workload} (bounded sample: {sample})"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": len(reqs), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_dry(args, world, rank):
    """--dry-run: the rank logic alone (gloo, no GPU): every rank joins, takes
    its request shard, and rank 0 prints who took part."""
    dist = init_dist(world, "gloo")
    barrier(dist)
    ranks = reduce_sum(dist, float(1 << rank))
    seeds = reduce_sum(dist, float(args.seed + rank))
    if rank == 0:
        print(json.dumps({"dry_run": True, "n_gpus": world, "rank_mask": int(ranks), "seed_sum": int(seeds)}),
              flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["dkv", "reference"], default="dkv")
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--decode-steps", type=int, default=None)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--extras", default="llama70b,llama8b@4096,qwen7b,llama8b+mid",
                    help="other configurations measured after the headline (workload[@page_bytes],...; 'none')")
    ap.add_argument("--extra-steps", type=int, default=2)
    ap.add_argument("--churn-ticks", type=int, default=1500,
                    help="ticks of the QwQ-32B-shaped arrival / completion workload (0: skip)")
    ap.add_argument("--prefill-reps", type=int, default=3,
                    help="timed repetitions of the prompt attention and prefilled compaction (0: skip)")
    ap.add_argument("--prefill-requests", type=int, default=None,
                    help="first N requests of the workload for the prefill part (default: all)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--dry-run", action="store_true", help="rank start-up and reductions only (gloo, no GPU)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu DRAM bytes per decode_attention launch, when known for the current kernel sources")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args.gpus))
    if args.decode_steps is None:
        args.decode_steps = workloads.WORKLOADS[args.workload].decode_steps
    world, rank, local = dist_env()
    if args.dry_run:
        run_dry(args, world, rank)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_dkv(args, world, rank, local)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the differentiated-KV hot path on GB300 (one process per GPU).

One step = one pass of the whole path over one batch of the Llama-3-8B-shaped
workload (32 requests x 4096-token prompts, 32 q / 8 KV heads):
  prompt compact_step (score, classify, grant, pack, reclaim)
  then 128 decode steps: [L2 flush] decode compact_step + decode_attention
  (with score update), then free_request for every request.
value = decode-attention GB/s: algorithmic bytes (hi token 200 B, lo token
104 B, +8 B score update, + q and out) over the device time of the
decode_attention calls (CUDA events on the launch stream, L2 flushed before
each call). compact_step is reported in us per layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dkv|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "compressed-KV decode attn GB/s (% of GB300 HBM peak); compact_step µs/layer"
HI_BYTES, LO_BYTES, SCORE_RMW = 200, 104, 8

# DRAM bytes of one decode-attention call (k_attn_paged + k_attn_epi:
# dram__bytes_read.sum + dram__bytes_write.sum, caches flushed by ncu before
# each kernel), third decode step of the llama8b bench step.
# Valid only for the kernel sources it was taken on: any change to them
# makes the bench report null until a new capture replaces the record.
ATTN_TRAFFIC = {
    "workload": "llama8b",
    "bytes_per_call": 119_673_600 + 8_354_304 + 25_937_664,
    "sources": {
        "attention.cu": "698d960b729c03922d29c7d9cfad8c6cd063d4b7bc8d69b31a1222a246023e03",
        "dkv_common.cuh": "90d758348e6dbf3a1ae34973ef9bef33cbbd31e8c1a636103b676ac54b52f649",
        "dkv_kernels.cuh": "a11e8c64feb0a4bcfea04df84fe718b26a0fa6dc53df45de115fabf6c95d12fe",
    },
}


def recorded_traffic(workload: str):
    """The recorded per-call DRAM traffic when the attention sources still
    hash to those it was captured on, else None."""
    if workload != ATTN_TRAFFIC["workload"]:
        return None
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "differentiated_kv_cache_gb300", "csrc")
    for name, digest in ATTN_TRAFFIC["sources"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return ATTN_TRAFFIC["bytes_per_call"]
L2_FLUSH_BYTES = 256 << 20


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
                                          "--format=csv,noheader,nounits", "-lms", "200"],
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


# --------------------------------------------------------------- workload
def load_inputs(name: str, seed: int, decode_steps: int):
    w = workloads.WORKLOADS[name]
    inp = workloads.prompt_inputs(name, seed)
    dec = [workloads.decode_inputs(name, t, seed) for t in range(decode_steps)]
    return w, inp, dec


def attn_bytes(hi_tokens: int, lo_tokens: int, n_req: int, hq: int, update: bool) -> int:
    per = HI_BYTES * hi_tokens + LO_BYTES * lo_tokens
    if update:
        per += SCORE_RMW * (hi_tokens + lo_tokens)
    return per + n_req * hq * (128 * 2 + 128 * 4)


def prompt_bytes(hi_tokens: int, lo_tokens: int, n_tokens_heads: int, n_req: int, hq: int) -> int:
    return 512 * n_tokens_heads + 208 * hi_tokens + 112 * lo_tokens + n_req * 32 * hq * 256


# ------------------------------------------------------------- dkv (GPU)
def run_dkv(args, world, rank, local):
    import torch
    import differentiated_kv_cache_gb300 as dkv
    dkv.build.build()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    w, inp, dec = load_inputs(args.workload, args.seed + rank, args.decode_steps)
    H, G, R = w.n_kv_heads, w.group_size, w.n_requests
    Hq = H * G
    lens = [int(x) for x in inp["lens"]]
    cfg = w.pool_config()
    cfg["max_seq_len"] = max(lens) + args.decode_steps
    pool = dkv.dkv_pool_create(dkv.make_config(**{k: v for k, v in cfg.items()
                                                   if k in dict(dkv.dkv_config._fields_)}), local)
    slots = list(range(R))
    # device-resident inputs
    k_d = torch.from_numpy(inp["k"]).to(dev)
    v_d = torch.from_numpy(inp["v"]).to(dev)
    q_d = torch.from_numpy(inp["q_obs"]).to(dev)
    dk = torch.from_numpy(np.stack([d["k"] for d in dec])).to(dev)
    dv = torch.from_numpy(np.stack([d["v"] for d in dec])).to(dev)
    dq = torch.from_numpy(np.stack([d["q"] for d in dec])).to(dev)
    out = torch.zeros((R, Hq, 128), dtype=torch.float32, device=dev)
    # L2 flush between decode steps: write a buffer larger than L2, then read a
    # second one so that the write-back of the dirty lines happens here and not
    # inside the next timed kernel; L2 then holds none of the path's data.
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    T = args.decode_steps

    def step(record=None, counts=None):
        """One pass of the path. record: dict of event lists; counts: list to
        fill with (hi, lo) stored tokens at each decode_attention (syncs)."""
        ev = lambda: torch.cuda.Event(enable_timing=True)
        if record is not None:
            e0, e1 = ev(), ev()
            e0.record(stream)
        dkv.dkv_compact_step(pool, 0, dkv.DKV_PROMPT, slots, lens, k_d, v_d, q_d)
        if record is not None:
            e1.record(stream)
            record["prompt"].append((e0, e1))
        if counts is not None:
            st = dkv.dkv_pool_status(pool)
            counts.append(("prompt", st["hi_tokens"], st["lo_tokens"]))
        for t in range(T):
            flush.fill_(t & 0xFF)
            torch.amax(flush_rd)
            # Even steps put an event between compaction and attention (the
            # compaction alone), odd steps do not: there the attention kernel
            # launches while the compaction drains, as in a decode loop, and
            # (compaction + attention) is timed as one.
            split = t % 2 == 0
            if record is not None:
                c0, c1, a1 = ev(), ev(), ev()
                c0.record(stream)
            dkv.dkv_compact_step(pool, 0, dkv.DKV_DECODE, slots, None, dk[t], dv[t])
            if record is not None and split:
                c1.record(stream)
            dkv.dkv_decode_attention(pool, 0, slots, dq[t], out, True)
            if record is not None:
                a1.record(stream)
                if split:
                    record["compact"].append((c0, c1))
                    record["attn_split"].append((c1, a1))
                else:
                    record["pair"].append((c0, a1))
            if counts is not None:
                st = dkv.dkv_pool_status(pool)
                counts.append(("attn", st["hi_tokens"], st["lo_tokens"]))
        for s in slots:
            dkv.dkv_free_request(pool, s)

    # warm-up; the first warm-up step also records the stored-token counts
    counts = []
    for i in range(max(args.warmup, 1)):
        step(counts=counts if i == 0 else None)
    torch.cuda.synchronize()
    st = dkv.dkv_pool_status(pool)
    assert st["error"] == 0, st
    prompt_counts = counts[0]
    attn_counts = [c for c in counts if c[0] == "attn"]
    bytes_per_attn = [attn_bytes(c[1], c[2], R, Hq, True) for c in attn_counts]
    n_th = sum(lens) * H
    pbytes = prompt_bytes(prompt_counts[1], prompt_counts[2], n_th, R, Hq)

    rec = {"prompt": [], "compact": [], "attn_split": [], "pair": []}
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            step(record=rec)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(dist)
    step_ms = t_start.elapsed_time(t_end) / args.steps
    compact_ms = [a.elapsed_time(b) for a, b in rec["compact"]]
    prompt_ms = [a.elapsed_time(b) for a, b in rec["prompt"]]
    pair_ms = [a.elapsed_time(b) for a, b in rec["pair"]]
    # a decode-attention call's time: (compaction + attention) of the odd
    # steps less the compaction alone of the even steps; with one decode step
    # only, the even step's attention after its event
    if pair_ms:
        call_ms = statistics.mean(pair_ms) - statistics.mean(compact_ms)
    else:
        call_ms = statistics.mean([a.elapsed_time(b) for a, b in rec["attn_split"]])
    attn_ms = [call_ms] * (T * args.steps)
    attn_total_ms = sum(attn_ms)
    attn_total_bytes = sum(bytes_per_attn) * args.steps
    step_ms_max = reduce_max(dist, step_ms, dev)
    attn_ms_max = reduce_max(dist, attn_total_ms, dev)
    all_bytes = reduce_sum(dist, attn_total_bytes, dev)
    value = all_bytes / (attn_ms_max * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    per_launch_bytes = sum(bytes_per_attn) / len(bytes_per_attn)
    per_launch_ms = attn_total_ms / len(attn_ms)
    achieved = per_launch_bytes / (per_launch_ms * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic (seeded numpy; model-shaped K/V/Q, no weights or datasets)",
        "config": {
            "workload": f"{w.name}: {w.shape or 'synthetic'}-shaped layer, {R} requests x "
                        f"{min(lens)}-{max(lens) if max(lens) != min(lens) else ''}".rstrip("-") +
                        f"-token prompts, {Hq} q / {H} KV heads, d=128, {T} decode steps with compaction and "
                        f"score update",
            "requests": R, "prompt_len": lens[0], "decode_steps": T, "q_heads": Hq, "kv_heads": H,
            "alpha_h": w.alpha_h, "alpha_l": w.alpha_l, "window": w.recent_window, "page_bytes": w.page_bytes,
            "l2": "flushed before every decode step, outside the timed events: 256 MiB written, then a "
                  "second 256 MiB read (L2 left clean); prompt inputs 537 MB > L2",
            "value_is": "decode-attention algorithmic bytes / decode_attention device time; a call's time is "
                        "(compaction + attention) timed as one on odd decode steps, where the attention kernel "
                        "launches while the compaction drains as in a decode loop, less the compaction alone "
                        "timed on even steps",
            "parallelism": f"{world} independent pools (one per GPU), no collective in the path",
        },
        "parts": {
            "compact_step_prompt_us_per_layer": round(statistics.mean(prompt_ms) * 1e3, 1),
            "compact_step_prompt_gbs": round(pbytes / (statistics.mean(prompt_ms) * 1e-3) / 1e9, 1),
            "compact_step_decode_us_per_layer": round(statistics.mean(compact_ms) * 1e3, 2),
            "decode_attention_us": round(statistics.mean(attn_ms) * 1e3, 2),
            "stored_tokens_after_prompt": {"hi": prompt_counts[1], "lo": prompt_counts[2],
                                           "pruned": n_th - prompt_counts[1] - prompt_counts[2]},
            "kv_bytes_vs_fp16": round((HI_BYTES * prompt_counts[1] + LO_BYTES * prompt_counts[2]) / (n_th * 512), 4),
        },
        "roofline": {"bound": "hbm", "kernel": "dkv_decode_attention call (k_attn_paged + k_attn_epi)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": int(per_launch_bytes),
                     "traffic": args.traffic if args.traffic is not None else recorded_traffic(args.workload)},
        # per step: prompt compact_step 11 kernels; per decode step 3 (compaction)
        # + 2 (attention, epilogue); one free_request kernel per request
        "gpu_launches": args.steps * (11 + T * 5 + R),
    }
    result["clocks"] = clk.summary()
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, dkv, pool, w, inp, dec, lens, slots, sum(bytes_per_attn), dev, dist)
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args)
    dkv.dkv_pool_destroy(pool)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, dkv, pool, w, inp, dec, lens, slots, attn_bytes_step, dev, dist):
    """The same step through the C ABI with inputs in pinned host memory:
    every step copies the prompt K/V/Q and each decode step's K/V/q to the
    device and reads each decode step's attention output back."""
    import torch
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hk, hv, hq = pin(inp["k"]), pin(inp["v"]), pin(inp["q_obs"])
    hdk = [pin(d["k"]) for d in dec]
    hdv = [pin(d["v"]) for d in dec]
    hdq = [pin(d["q"]) for d in dec]
    R, Hq = w.n_requests, w.n_q_heads
    hout = torch.empty((R, Hq, 128), dtype=torch.float32).pin_memory()
    k_d = torch.empty(hk.shape, dtype=torch.float16, device=dev)
    v_d = torch.empty_like(k_d)
    q_d = torch.empty(hq.shape, dtype=torch.float16, device=dev)
    dk = torch.empty(hdk[0].shape, dtype=torch.float16, device=dev)
    dv = torch.empty_like(dk)
    dq = torch.empty(hdq[0].shape, dtype=torch.float16, device=dev)
    out = torch.empty((R, Hq, 128), dtype=torch.float32, device=dev)
    T = args.decode_steps

    def step():
        k_d.copy_(hk, non_blocking=True); v_d.copy_(hv, non_blocking=True); q_d.copy_(hq, non_blocking=True)
        dkv.dkv_compact_step(pool, 0, dkv.DKV_PROMPT, slots, lens, k_d, v_d, q_d)
        for t in range(T):
            dk.copy_(hdk[t], non_blocking=True); dv.copy_(hdv[t], non_blocking=True)
            dq.copy_(hdq[t], non_blocking=True)
            dkv.dkv_compact_step(pool, 0, dkv.DKV_DECODE, slots, None, dk, dv)
            dkv.dkv_decode_attention(pool, 0, slots, dq, out, True)
            hout.copy_(out, non_blocking=True)
        for s in slots:
            dkv.dkv_free_request(pool, s)
        torch.cuda.synchronize()

    step()
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    dt = reduce_max(dist, dt, dev)
    n = dist.get_world_size() if dist is not None else 1
    h2d = hk.numel() * 2 + hv.numel() * 2 + hq.numel() * 2 + T * (hdk[0].numel() + hdv[0].numel() + hdq[0].numel()) * 2
    d2h = T * hout.numel() * 4
    return {"value": round(n * attn_bytes_step / dt / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(dt * 1e3, 2),
            "what": "decode-attention algorithmic bytes of a step / wall time of the whole step through the "
                    "C ABI from pinned host buffers (host sync at the end of each step)"}


# --------------------------------------------------- oracle (CPU baseline)
def oracle_sample(name: str, seed: int, n_decode: int):
    """The oracle as it stands on a bounded sample of the workload: one
    request's prompt compaction (fp64 scoring) and n_decode decode steps
    (compaction + fp64 attention with score update). Returns
    (attention bytes, attention seconds, prompt seconds per layer-request)."""
    import oracle
    w = workloads.WORKLOADS[name]
    inp = workloads.prompt_inputs(name, seed, requests=[0])
    cfg = w.pool_config(max_requests=1, max_seq_len=int(inp["lens"][0]) + n_decode, n_pages=
                        2 * w.n_kv_heads * (int(inp["lens"][0]) // 18 + n_decode + 8))
    pool = oracle.Pool(cfg)
    t0 = time.perf_counter()
    rc = pool.prompt(0, [0], inp["lens"], inp["k"], inp["v"], inp["q_obs"])
    tp = time.perf_counter() - t0
    assert rc == 0
    ab, at = 0, 0.0
    for t in range(n_decode):
        d = workloads.decode_inputs(name, t, seed, requests=[0])
        assert pool.decode(0, [0], d["k"], d["v"]) == 0
        hc = pool.head_counts[0, 0]
        hi, lo = int(hc[:, 0].sum()), int(hc[:, 1].sum())
        t0 = time.perf_counter()
        rc, _ = pool.attention(0, [0], d["q"], update_scores=True)
        at += time.perf_counter() - t0
        ab += attn_bytes(hi, lo, 1, w.n_q_heads, True)
    return ab, at, tp


def cpu_baseline(args) -> dict:
    n_dec = 16
    ab, at, tp = oracle_sample(args.workload, args.seed, n_dec)
    return {"value": round(ab / at / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"1 of 32 requests (4096-token prompt, 8 KV heads), {n_dec} decode steps; "
                      f"prompt compact_step of that request {tp * 1e3:.0f} ms (fp64 scoring)",
            "compact_step_prompt_us_per_request_layer": round(tp * 1e6, 0)}


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    n_dec = 8
    for _ in range(args.warmup):
        oracle_sample(args.workload, args.seed, 1)
    tot_b, tot_t, t_all = 0, 0.0, 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ab, at, tp = oracle_sample(args.workload, args.seed, n_dec)
        tot_b += ab
        tot_t += at
    t_all = time.perf_counter() - t0
    value = tot_b / tot_t / 1e9
    sample = f"1 of 32 requests (4096-token prompt, 8 KV heads), {n_dec} decode steps per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_all / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.workload} (bounded sample: {sample})"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["dkv", "reference"], default="dkv")
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--decode-steps", type=int, default=None)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu DRAM bytes per decode_attention launch, when known for this build")
    args = ap.parse_args()
    if args.decode_steps is None:
        args.decode_steps = workloads.WORKLOADS[args.workload].decode_steps
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_dkv(args, world, rank, local)


if __name__ == "__main__":
    main()

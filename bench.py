#!/usr/bin/env python
"""MLA decode benchmark on B300: prints one JSON line.

One step = one pass of the whole hot path over the workload's batch:
compress + RoPE + paged append of the T new tokens of every sequence, then
the absorbed decode (query absorption, split-KV attention, combine, W^UV,
W_O), replayed as one CUDA graph.  Inputs and state are resident in HBM
when the timed region starts; L2 is flushed (a 2x-L2 buffer is written,
then another is read) before every timed step, outside the step's own
CUDA-event bracket.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config b128-l16k-t2]
                  [--impl mla|reference]

The default workload is the full layer step at DeepSeek-V2 widths (batch
128, 16384 cached tokens, two query tokens): the largest single-GPU
workload, on which the throughput metric is quoted.

--impl reference times the fp64 CPU oracle (the reference of this build)
on the same workload, a bounded sample per step.  Under torchrun (N > 1)
every rank runs an independent replica on its own GPU (the step has no
cross-GPU exchange); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s and latent-cache GB/s (% of B300 roofline), 1 GPU"
METRIC_PREFILL = "MLA prefill tokens/s (a causal chunk of T new tokens per sequence), 1 GPU"
DEFAULT_STEPS = {"tiny-fp32": 200, "b1-l4096": 1000, "b64-paged": 300, "b4-l128k": 300,
                 "b128-l16k-t2": 50, "b1-l4096-x60": 30, "b64-paged-x8": 30,
                 "prefill-b4-t4096": 20, "chunk-b1-l12k-t4096": 20, "prefill-b64-t128": 50}
PREFILL = ("prefill-b4-t4096", "chunk-b1-l12k-t4096", "prefill-b64-t128")
FORMS = {"auto": 0, "explicit": 1, "absorbed": 2}


# ----------------------------------------------------------------------------- setup
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="b128-l16k-t2",
                    choices=["tiny-fp32", "b1-l4096", "b64-paged", "b4-l128k", "b128-l16k-t2",
                             "b1-l4096-x60", "b64-paged-x8"] + list(PREFILL))
    ap.add_argument("--kv", default="native", choices=["native", "fp8"],
                    help="latent-cache storage: the context dtype, or E4M3 rows of 656 bytes "
                         "(bf16 workloads)")
    ap.add_argument("--form", default="auto", choices=list(FORMS),
                    help="prefill workloads: the attention form mla_prefill uses (auto: the "
                         "library's choice by FLOPs)")
    ap.add_argument("--impl", default="mla", choices=["mla", "reference"])
    ap.add_argument("--query-path", action="store_true",
                    help="time the step from the hidden states alone (mla_layer_step: the "
                         "query projections W^DQ, W^UQ, W^QR, then append and decode)")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling cut: keep the first N sequences of the workload")
    ap.add_argument("--cache-len", type=int, default=0,
                    help="profiling cut: every sequence holds this many cached tokens")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    a = ap.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.config]
    a.warmup = max(a.warmup, 3)
    if a.config.endswith(("-x60", "-x8")):
        a.query_path = True   # a layer stack makes every layer's queries from its input
    return a


def dist_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def sources_hash(files) -> str:
    """sha256 (16 hex digits) of the named files under the package's csrc/."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(files):
        h.update(name.encode())
        with open(os.path.join(ROOT, "mla_latent_kv_82_b300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def captured_traffic(config_key: str, kernel: str):
    """DRAM bytes per launch of `kernel` on workload `config_key` from the
    committed ncu summary, if the kernel's sources still hash as they did
    when it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(config_key, {}).get(kernel)
        if not rec or rec.get("sources_sha256_16") != sources_hash(rec["sources"]):
            return None
    except (OSError, ValueError, KeyError):
        return None
    return rec["dram_bytes"]


# ----------------------------------------------------------------------------- work model
def work_model(wl, query_path=False, form="absorbed", kv="native"):
    """Algorithmic bytes and FLOPs per launch of each kernel, and per step.

    form="explicit": a prefill chunk in the explicit form (gather the cached
    rows, up-project K^C and V per head, causal attention over 192 + 128
    features, W_O); otherwise the absorbed decode kernels."""
    d = wl.dims
    es = 2 if wl.dtype == "bf16" else 4
    M, H, dc, dr, R = wl.B * wl.T, d.n_heads, d.d_latent, d.d_rope, d.row_width
    dn, dv, D = d.d_nope, d.d_v, d.d_model
    cache_rows = sum(wl.seq_lens)
    visible = sum(S - wl.T + t + 1 for S in wl.seq_lens for t in range(wl.T))
    k = {
        "compress_append": (R * D * es + M * D * es + M * R * es, 2.0 * M * R * D),
        "absorb_q": (H * dn * dc * es + M * H * (dn + dr) * es + M * H * R * es,
                     2.0 * M * H * dn * dc),
        "attend": (cache_rows * R * es + M * H * R * es, 2.0 * visible * H * (R + dc)),
        "combine": (M * H * dc * es, 0.0),
        "value_proj": (H * dv * dc * es + M * H * dc * es + M * H * dv * es,
                       2.0 * M * H * dv * dc),
        "combine_uv": (H * dv * dc * es + M * H * dv * es, 2.0 * M * H * dv * dc),
        "out_proj": (D * H * dv * es + M * H * dv * es + M * D * es, 2.0 * M * D * H * dv),
        "plan": (wl.B * 4, 0.0),
    }
    if form == "explicit":
        n = cache_rows
        k.update({
            "gather": (2 * n * R * es, 0.0),
            "key_up": (H * dn * dc * es + n * dc * es + n * H * dn * es, 2.0 * n * H * dn * dc),
            "value_up": (H * dv * dc * es + n * dc * es + n * H * dv * es,
                         2.0 * n * H * dv * dc),
            "rope_q": (2 * M * H * (dn + dr) * es, 0.0),
            "prefill_attend": (M * H * (dn + dr) * es + n * (H * (dn + dv) + dr) * es
                               + M * H * dv * es, 2.0 * visible * H * (dn + dr + dv)),
        })
        steps = ["compress_append", "gather", "key_up", "value_up", "rope_q", "prefill_attend",
                 "out_proj"]
        return (k, sum(k[x][0] for x in steps), sum(k[x][1] for x in steps),
                cache_rows * R * es)
    # one launch runs the append and the absorbed query together
    k["append_absorb"] = tuple(a + b for a, b in zip(k["compress_append"], k["absorb_q"]))
    tot_bytes = (R * D + H * dn * dc + H * dv * dc + D * H * dv) * es \
        + cache_rows * R * es + M * (D + H * (dn + dr) + D) * es
    steps = ["compress_append", "absorb_q", "attend", "value_proj", "out_proj"]
    if query_path:
        cq = d.d_cq
        k["query_down"] = (cq * D * es + M * D * es + M * cq * es, 2.0 * M * cq * D)
        k["query_rope"] = (H * dr * D * es + M * D * es + M * H * dr * es, 2.0 * M * H * dr * D)
        k["query_up"] = (H * dn * cq * es + M * cq * es + M * H * dn * es, 2.0 * M * H * dn * cq)
        # the queries are no longer an input: their weights are read instead
        tot_bytes += (cq * D + H * dn * cq + H * dr * D) * es - M * H * (dn + dr) * es
        steps += ["query_down", "query_rope", "query_up"]
    if kv == "fp8":
        # E4M3 rows of 656 bytes in place of 576 bf16 values; the append
        # stages bf16 rows that f8_prepare quantises, with the query images
        R8, Q8 = 656, 82432
        k["f8_prepare"] = (M * R * es + M * R8 + M * H * R * es + M * Q8, 0.0)
        k["attend"] = (cache_rows * R8 + M * Q8, 2.0 * visible * H * (R + dc))
        tot_bytes += cache_rows * (R8 - R * es) + k["f8_prepare"][0]
        steps.append("f8_prepare")
    tot_flops = sum(k[n][1] for n in steps)
    if wl.layers > 1:
        # every layer reads its own weights and cache; the residual reads h and
        # u and writes h; the queries and new rows of layers > 0 come from h
        k["residual"] = (3 * M * D * es, 1.0 * M * D)
        tot_bytes = (tot_bytes + k["residual"][0]) * wl.layers
        tot_flops = (tot_flops + k["residual"][1]) * wl.layers
        return k, tot_bytes, tot_flops, cache_rows * (656 if kv == "fp8" else R * es) * wl.layers
    return k, tot_bytes, tot_flops, cache_rows * (656 if kv == "fp8" else R * es)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, bus_id):
        self.samples = []
        self.proc = None
        self.bus_id = bus_id

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.bus_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "during the timed region"
        if not win:
            win = [s for s in self.samples if t0 - 1.0 <= s[0] <= t1 + 1.0]
            note = "within 1 s of the timed region (region shorter than the sampling period)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi gave no samples"}
        sm = sorted(v for v in (num(p[0]) for _, p in win) if v is not None)
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in win:
            for n, v in zip(names, p[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": num(win[0][1][1]),
                "power_w_max": max((num(p[2]) or 0.0) for _, p in win),
                "reasons": sorted(reasons), "samples": len(win), "note": note}


# ----------------------------------------------------------------------------- oracle timing
def oracle_sample_setup(wl, device):
    """fp64 state for timing the oracle on one sequence (b = 0), untimed."""
    import numpy as np
    import torch
    from oracle import case as ocase
    from oracle import mla as omla
    names = ("w_dkv", "w_kr", "w_uk", "w_uv", "w_o") + \
        (("w_dq", "w_uq", "w_qr") if wl.dims.d_cq and wl.layers > 1 else ())
    w64 = ocase.weights_f64(wl, names=names, device=device)
    L = wl.lens[0]
    rows = np.empty((L, wl.dims.row_width))
    for p0 in range(0, L, 8192):
        p1 = min(L, p0 + 8192)
        h = wl.h_rows(0, p0, p1, device=device).to(torch.float64).cpu().numpy()
        rows[p0:p1] = omla.latent_rows(h, w64["w_dkv"], w64["w_kr"], np.arange(p0, p1),
                                       wl.dims.rope_base)
    h_new = wl.h_rows(0, L, L + wl.T, device=device).to(torch.float64).cpu().numpy()
    if wl.layers > 1:   # layer 0 of the stack: queries from the query path
        q64 = omla.query_from_hidden(wl.dims, h_new, w64["w_dq"], w64["w_uq"], w64["w_qr"])
    else:
        q64 = wl.q(device=device)[0].to(torch.float64).cpu().numpy()
    return {"w": w64, "rows": rows, "h_new": h_new, "q": q64}


def oracle_sample_step(wl, st, head):
    """One oracle decode step of sequence 0 restricted to one head.

    The unmodified oracle functions run on the head's slices of W^UK, W^UV
    and W_O (its contribution to u); the new tokens' rows are appended first.
    """
    import numpy as np
    from oracle import mla as omla
    d = wl.dims
    L = wl.lens[0]
    new = omla.latent_rows(st["h_new"], st["w"]["w_dkv"], st["w"]["w_kr"],
                           np.arange(L, L + wl.T), d.rope_base)
    rows = np.concatenate([st["rows"], new])
    w = {"w_uk": st["w"]["w_uk"][head * d.d_nope:(head + 1) * d.d_nope],
         "w_uv": st["w"]["w_uv"][head * d.d_v:(head + 1) * d.d_v],
         "w_o": st["w"]["w_o"][:, head * d.d_v:(head + 1) * d.d_v]}
    one = dataclasses.replace(d, n_heads=1)
    return omla.decode_explicit(one, rows, st["q"][:, head:head + 1], w, wl.T)["u"]


def time_oracle(wl, st, steps=None, seconds=None):
    """Returns (tokens/s, seconds timed, steps timed, sample description)."""
    H = wl.dims.n_heads
    per_step_tokens = wl.T / (H * wl.layers)   # one head of one layer of one sequence
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_sample_step(wl, st, n % H)
        n += 1
        el = time.perf_counter() - t0
        if steps is not None and n >= steps:
            break
        if seconds is not None and el >= seconds:
            break
    lay = f" of layer 0 of {wl.layers}" if wl.layers > 1 else ""
    sample = (f"sequence 0 (cache {wl.lens[0]} + {wl.T} new tokens), one of {H} heads{lay} per "
              f"step, explicit fp64 form incl. the new rows' W^DKV/W^KR; tokens/s = "
              f"T/({H}*{wl.layers}) per step / step time")
    return per_step_tokens * n / el, el, n, sample


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest of every rank's x (the slowest rank's time); x at N = 1."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: int, steps: int, world: int, total_ms: float) -> float:
    """Units all ranks processed per second over the slowest rank's time."""
    return units_per_rank_step * steps * world / (total_ms * 1e-3)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------------------- arms
def run_reference(a, wl, rank, world):
    if rank != 0:
        return None
    st = oracle_sample_setup(wl, "cpu" if not _cuda() else "cuda:0")
    for _ in range(a.warmup):
        oracle_sample_step(wl, st, 0)
    tps, el, n, sample = time_oracle(wl, st, steps=a.steps)
    return {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": 1e3 * el / n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "batch": wl.B, "T": wl.T},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _cuda():
    import torch
    return torch.cuda.is_available()


def run_mla(a, wl, rank, local_rank, world):
    prefill = a.config in PREFILL
    import torch
    import torch.distributed as dist
    import mla_latent_kv_82_b300 as m
    from mla_latent_kv_82_b300.workload import DeviceState

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    if wl.layers > 1:
        from mla_latent_kv_82_b300.workload import StackState
        st = StackState(wl, device=local_rank)
        step = st.step
    else:
        st = DeviceState(wl, device=local_rank, query_path=a.query_path, kv=a.kv)
        step = st.layer_step if a.query_path else st.step
        if prefill:
            form = FORMS[a.form]
            step = lambda: st.prefill_chunk(form)   # noqa: E731
            step()   # sizes the prefill workspace outside the captured graph
    torch.cuda.synchronize()
    l2 = getattr(props, "L2_cache_size", 126 << 20) or (126 << 20)
    # L2 flush: write a 2x-L2 buffer, then read another one, so the timed step
    # starts with a cold L2 that holds no dirty lines to write back
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=sink)

    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    check_status = st.check_status if wl.layers > 1 else st.mla.check_status
    launch_count = (lambda: sum(m.launch_count() for m in st.mlas)) if wl.layers > 1 \
        else st.mla.launch_count
    prof_ctxs = [m.ctx for m in st.mlas] if wl.layers > 1 else [st.mla.ctx]
    if check_status() != 0:
        raise RuntimeError("device status set during warm-up")

    # one decode step (append + decode) as a CUDA graph, replayed every step
    n0 = launch_count()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        step()
    launches_per_step = launch_count() - n0
    for _ in range(a.warmup):
        flush()
        g_step.replay()
    torch.cuda.synchronize()

    bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0" \
        if hasattr(props, "pci_bus_id") else str(local_rank)
    clocks = ClockSampler(bus)
    clocks.start()
    time.sleep(0.3)
    stream = torch.cuda.current_stream()

    # ---- timed region: K steps, each bracketed by CUDA events, flush outside
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(a.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(a.steps):
        flush()
        evs[i][0].record(stream)
        g_step.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    step_ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in evs), dev)
    status = check_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    time.sleep(0.2)
    clocks.stop()
    launches = launches_per_step * a.steps

    value = whole_job_rate(wl.B * wl.T, a.steps, world, step_ms)
    ms_per_step = step_ms / a.steps

    # ---- per-kernel durations: the same steps with an event at every kernel
    # boundary (events keep kernels from overlapping, so this pass only
    # apportions time between kernels; the step time comes from the pass above)
    for cx in prof_ctxs:
        m.mla_profile_enable(cx, 1)
    g_prof = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_prof):
        step()
    kt = {}
    for i in range(a.steps):
        flush()
        g_prof.replay()
        for cx in prof_ctxs:
            for name, ms in m.mla_profile_read(cx):
                kt.setdefault(name, []).append(ms)
    for cx in prof_ctxs:
        m.mla_profile_enable(cx, 0)

    # ---- roofline of the dominant kernel and of the whole step
    resolved = "explicit" if "prefill_attend" in kt else "absorbed"
    kmodel, tot_bytes, tot_flops, cache_bytes = work_model(wl, a.query_path, resolved, a.kv)
    avg = {k: sum(v) / len(v) for k, v in kt.items() if v}
    share = {k: sum(v) for k, v in kt.items()}
    dom = max(share, key=share.get)
    b_dom, f_dom = kmodel[dom]
    t_dom = avg[dom] * 1e-3
    bw_peak = peaks["hbm_gbs"]
    tf_peak = peaks["bf16_tflops"]
    mem_bound = (b_dom / (bw_peak * 1e9)) >= (f_dom / (tf_peak * 1e12)) or wl.dtype != "bf16"
    if mem_bound:
        roof = {"bound": "hbm", "achieved": b_dom / t_dom / 1e9, "peak": bw_peak,
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": f_dom / t_dom / 1e12, "peak": tf_peak,
                "unit": "TFLOP/s"}
    roof.update({"frac": roof["achieved"] / roof["peak"], "kernel": dom,
                 "traffic": None if (a.batch or a.cache_len) else
                 captured_traffic(a.config + ("+fp8" if a.kv == "fp8" else ""), dom),
                 "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json)"
                 if peaks["source"] == "measured" else "fallback",
                 "algorithmic_bytes_per_launch": b_dom, "algorithmic_flops_per_launch": f_dom,
                 "avg_launch_ms": avg[dom],
                 "timing": "per-kernel CUDA events on the launching stream, second pass of "
                           "the same steps"})
    t_step = ms_per_step * 1e-3
    step_roof = max(tot_bytes / (bw_peak * 1e9), tot_flops / (tf_peak * 1e12))

    # ---- end to end through the public API from pinned host buffers
    e2e = None
    if not a.no_e2e:
        # the step's inputs (new hidden states, queries, positions, lengths)
        # sit in one pinned staging buffer and go over in one copy
        dev_in = st.h0 if wl.layers > 1 else st.step_inputs
        dev_out = st.h if wl.layers > 1 else st.out
        in_h = dev_in.cpu().pin_memory()
        h2d = in_h.numel() * in_h.element_size()
        d2h = dev_out.numel() * dev_out.element_size()
        if world > 1:
            dist.barrier()
        if tot_bytes > l2:
            # The step reads more than L2 holds, so no flush is needed between
            # steps, and the copies of one step overlap the compute of the
            # one before, as a serving loop runs them: step k+1's inputs go
            # over on a copy stream while step k computes; each step then
            # moves its inputs from a device staging buffer into place, and
            # its output to a staging buffer that the copy stream reads back.
            xs = torch.cuda.Stream()
            stage_in = [torch.empty_like(dev_in) for _ in range(2)]
            stage_out = [torch.empty_like(dev_out) for _ in range(2)]
            out_h = [torch.empty(dev_out.shape, dtype=dev_out.dtype).pin_memory()
                     for _ in range(2)]
            K = a.steps
            ev_h2d = [torch.cuda.Event() for _ in range(K)]
            ev_in_used = [torch.cuda.Event() for _ in range(K)]
            ev_out = [torch.cuda.Event() for _ in range(K)]
            ev_d2h = [torch.cuda.Event() for _ in range(K)]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

            def upload(k):
                with torch.cuda.stream(xs):
                    if k >= 2:
                        xs.wait_event(ev_in_used[k - 2])   # staging buffer read by step k - 2
                    stage_in[k % 2].copy_(in_h, non_blocking=True)
                    ev_h2d[k].record(xs)

            torch.cuda.synchronize()
            e0.record(stream)
            xs.wait_event(e0)
            upload(0)
            for k in range(K):
                if k + 1 < K:
                    upload(k + 1)
                stream.wait_event(ev_h2d[k])
                dev_in.copy_(stage_in[k % 2], non_blocking=True)
                ev_in_used[k].record(stream)
                g_step.replay()
                if k >= 2:
                    stream.wait_event(ev_d2h[k - 2])      # output staging read back
                stage_out[k % 2].copy_(dev_out, non_blocking=True)
                ev_out[k].record(stream)
                with torch.cuda.stream(xs):
                    xs.wait_event(ev_out[k])
                    out_h[k % 2].copy_(stage_out[k % 2], non_blocking=True)
                    ev_d2h[k].record(xs)
            stream.wait_event(ev_d2h[K - 1])
            e1.record(stream)
            torch.cuda.synchronize()
            e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
            e2e_note = ("every step copies its inputs (one packed pinned buffer: new hidden "
                        "states, queries, positions, lengths) from host memory and its output "
                        "back; all inside the timed region, the copies of a step overlapping the "
                        "compute of the one before (copy stream, double-buffered device "
                        "staging); the step reads more than L2 holds, so no flush between steps")
        else:
            out_h = torch.empty(dev_out.shape, dtype=dev_out.dtype).pin_memory()

            def e2e_step():
                dev_in.copy_(in_h, non_blocking=True)
                step()
                out_h.copy_(dev_out, non_blocking=True)

            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e):
                e2e_step()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(a.steps)]
            torch.cuda.synchronize()
            for i in range(a.steps):
                flush()
                ev[i][0].record(stream)
                g_e2e.replay()
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            e_ms = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in ev), dev)
            e2e_note = ("every step copies its inputs (one packed pinned buffer: new hidden "
                        "states, queries, positions, lengths) from host memory and its output "
                        "back inside the timed region (one CUDA graph per step, L2 flushed "
                        "before each)")
        if check_status() != 0:
            raise RuntimeError("device status set during the end-to-end steps")
        e2e = {"value": whole_job_rate(wl.B * wl.T, a.steps, world, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "note": e2e_note}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        ost = oracle_sample_setup(wl, f"cuda:{local_rank}")
        tps, el, n, sample = time_oracle(wl, ost, seconds=a.cpu_seconds)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": sample + f"; {n} steps in {el:.1f} s"}

    if rank != 0:
        return None
    if prefill:
        graph = (f"each step is one CUDA-graph replay of mla_prefill (form {a.form}: "
                 f"{resolved} ran): append the chunk's rows, then causal attention and W_O")
    elif wl.layers > 1:
        graph = ("each step is one CUDA-graph replay of mla_multi_layer_step "
                 f"through {wl.layers} layers (each: queries from its input, "
                 "append, decode, residual)")
    elif a.query_path:
        graph = ("each step is one CUDA-graph replay of mla_layer_step (queries "
                 "from the new hidden states, append, decode)")
    else:
        graph = ("each step is one CUDA-graph replay of mla_append_decode "
                 "(append the new rows, then decode them)")
    return {
        "metric": METRIC_PREFILL if prefill else METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic: seeded N(0,1) hidden states and queries, N(0,1/fan_in) weights",
        "config": {"workload": wl.name + ("+query-path" if a.query_path and wl.layers == 1
                                          else ""),
                   "batch": wl.B, "T": wl.T, "layers": wl.layers,
                   **({"form": a.form, "form_ran": resolved} if prefill else {}),
                   "kv": "E4M3 rows of 656 bytes (per-row scale)" if a.kv == "fp8"
                         else "rows in the context dtype",
                   "cache_tokens": sum(wl.seq_lens), "l2": "flushed before every timed step "
                   f"(write {2 * l2 >> 20} MiB, then read {2 * l2 >> 20} MiB; outside the "
                   "step's event bracket)",
                   "graph": graph,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "cache_gbs": cache_bytes / t_step / 1e9,
                   "step_algorithmic_gb": tot_bytes / 1e9,
                   "step_algorithmic_gflop": tot_flops / 1e9,
                   "step_roofline_frac": step_roof / t_step,
                   "kernel_ms": {k: round(v, 5) for k, v in avg.items()},
                   "kernel_ms_note": "per-kernel times come from a second pass with a CUDA "
                                     "event at every kernel boundary (events keep kernels from "
                                     "overlapping, so they sum to more than ms_per_step, which is "
                                     "timed without them); kernel_share is their ratio",
                   "kernel_share": {k: round(v / sum(share.values()), 4) for k, v in share.items()}},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }


def main():
    a = parse()
    rank, local_rank, world = dist_info()
    from synth import workloads as W
    wl = W.config(a.config)
    if a.batch or a.cache_len:
        # a smaller case of the same shapes (for profiler captures; not a
        # benchmark line of the named workload)
        lens = wl.lens[:a.batch] if a.batch else wl.lens
        if a.cache_len:
            lens = [a.cache_len] * len(lens)
        wl = dataclasses.replace(wl, name=f"{wl.name}-cut-b{len(lens)}" +
                                 (f"-l{a.cache_len}" if a.cache_len else ""), lens=list(lens))
    if world > 1:
        import torch
        import torch.distributed as dist
        if a.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        res = run_reference(a, wl, rank, world) if a.impl == "reference" \
            else run_mla(a, wl, rank, local_rank, world)
    finally:
        if world > 1 and a.impl != "reference":
            import torch.distributed as dist
            dist.destroy_process_group()
    if res is not None and rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

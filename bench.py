"""Benchmark of the WeDLM window decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload low_entropy|full_stack|one_layer|ragged|tiny|...]
                    [--extra full_stack,one_layer,ragged | --extra none]

A step is one pass of the whole hot path (reorder + embed, every decoder
layer with paged window attention, LM head with streaming softmax, Eq. 11
selection, commit and refill) over one batch of synthetic input.  The
headline workload is the largest single-GPU one: the 36-layer
Qwen3-8B-shaped random-init bf16 stack in the low-entropy long-context
regime (prefix 32768, W=32, batch 8, a planted peaked next-token
distribution on a seeded counting sequence), streaming from an all-masked
window.  The other workloads (`--extra`) are measured after it, each with
its own roofline, and reported under "extra".

Prints ONE JSON line (rank 0).  `value` = committed tokens/s over the timed
steps (inputs resident in HBM; each step moves far more than the 129 MB L2,
so no flush is needed); `e2e` = the same metric through the Python API with
the window copied from pinned host memory and the results read back every
step.  The multi-GPU path runs independent replicas (one process per GPU, no
collective): `value` sums the tokens all ranks committed over the max time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth import WORKLOADS, make_state_np, plant_bias_for, plant_targets  # noqa: E402


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="low_entropy",
                    choices=["full_stack", "low_entropy", "one_layer", "ragged", "tiny",
                             "two_layer", "two_layer_long", "one_layer_long"])
    ap.add_argument("--extra", default="full_stack,one_layer,ragged,dual_stream,sweep",
                    help="comma-separated workloads measured after the headline one "
                         "('none' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def extras_all(args):
    return [e for e in args.extra.split(",") if e and e != "none"]


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def reduce_over_ranks(ms, committed, world, device):
    """Whole-job numbers of independent replicas: the slowest rank's time and
    the tokens every rank committed (no collective touches the data path;
    this is the only exchange, after the timed region)."""
    if world <= 1:
        return ms, committed
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, committed], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), int(sm[1])


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def load_tc_sustained():
    """bf16 tensor peak for kernels timed inside a long step (TFLOP/s)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        if "bf16_tflops_sustained" in d:
            return d["bf16_tflops_sustained"], "measured"
    return 1700.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes per launch of each kernel kind (HBM roofline units)
# ---------------------------------------------------------------------------
def algorithmic_bytes(shape, B, W, prefix_total):
    s = shape
    es = 2 if s.dtype == "bf16" else 4
    M = B * W
    H, hd, nq, nkv, F, V = s.hidden, s.head_dim, s.n_q_heads, s.n_kv_heads, s.ffn, s.vocab
    qkv_rows = (nq + 2 * nkv) * hd
    return {
        "gemm_qkv": es * (qkv_rows * H + M * H + M * qkv_rows),
        "gemm_o": es * (H * nq * hd + M * nq * hd + 2 * M * H),
        "gemm_gateup": es * (2 * F * H + M * H + M * F),
        "gemm_down": es * (H * F + M * F + 2 * M * H),
        "lmhead": es * (V * H + M * H),
        # every cached K/V byte once + window K/V + q in + o out
        "attn": es * (prefix_total * 2 * nkv * hd + B * W * 2 * nkv * hd + 2 * M * nq * hd),
    }


def algorithmic_flops(shape, B, W, prefix_total, masked_rows):
    """Tensor-core FLOPs per launch of each kind (two per multiply-add): the
    projections over all B*W rows, the LM head over the masked rows only,
    the attention over every visible (query row, key) pair, QK^T and P.V
    (4*hd per pair and q head; a window row at physical p sees its
    sequence's prefix and window rows 0..p)."""
    s = shape
    M = B * W
    H, hd, nq, nkv, F, V = s.hidden, s.head_dim, s.n_q_heads, s.n_kv_heads, s.ffn, s.vocab
    pairs = W * prefix_total + B * W * (W + 1) // 2
    return {
        "gemm_qkv": 2 * M * H * (nq + 2 * nkv) * hd,
        "gemm_o": 2 * M * nq * hd * H,
        "gemm_gateup": 2 * M * H * 2 * F,
        "gemm_down": 2 * M * F * H,
        "lmhead": int(2 * masked_rows * V * H),
        "attn": 4 * nq * hd * pairs,
    }


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms (a timed region
    of 20 steps at ~13 ms is about 260 ms)."""

    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [l.split(",") for l in open(self.f.name).read().splitlines() if l.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload set-up on the device
# ---------------------------------------------------------------------------
def setup(wl_name, steps, warmup, device, weights=None, loop_steps=0):
    from synth import make_pool_torch, make_weights_torch
    import dataclasses
    wl = WORKLOADS[wl_name]
    s = wl.shape
    extra = int(math.ceil((steps + warmup + 40 + loop_steps) * wl.window / s.page_block)) + 1
    wl = dataclasses.replace(wl, extra_pages=extra)
    st = make_state_np(wl)
    w = weights if weights is not None else make_weights_torch(s, seed=wl.seed, device=device)
    pools = [make_pool_torch(s, st["num_pages"], wl.seed, l, device=device)
             for l in range(s.n_layers)]
    plant = None
    if wl.plant:
        plant = plant_targets(st["pos"], s0=17)
    return wl, st, w, pools, plant


def _blas_threads():
    """Threads of the BLAS NumPy loaded: threadpoolctl when installed, else
    the OpenBLAS library mapped into this process, asked directly."""
    try:
        from threadpoolctl import threadpool_info
        return max(int(i.get("num_threads", 1)) for i in threadpool_info()
                   if i.get("user_api") == "blas")
    except Exception:
        pass
    import ctypes
    try:
        libs = {l.split()[-1] for l in open("/proc/self/maps") if "openblas" in l.lower()}
    except OSError:
        libs = set()
    for path in sorted(libs):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                    "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
            f = getattr(lib, sym, None)
            if f is not None:
                return int(f())
    return None


def host_info():
    """CPU model, core count and the BLAS threads NumPy uses."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"cpu": model, "cores": os.cpu_count(), "blas_threads": _blas_threads()}


def cpu_sample(wl, w, st, ctx_commits_per_step):
    """Time the oracle (as it stands) on a bounded sample of one step: one
    decoder layer over one sequence's window, the LM head over 2 rows and
    the selection of one sequence, then scale to the whole step (all layers,
    all sequences, all rows).  The returned step time is an extrapolation
    from that sample, and the record says so."""
    import oracle as O
    s = wl.shape
    W = wl.window
    lw = {k: v.float().cpu().numpy() for k, v in w["layers"][0].items()}
    lm = w["lm_head"].float().cpu().numpy()
    norm = w["final_norm"].float().cpu().numpy()
    rng = np.random.default_rng(0)
    x = O.bf16_round(rng.standard_normal((W, s.hidden)) * 0.05)
    L = int(st["seq_len"][0])
    kp = O.bf16_round(rng.standard_normal((L, s.n_kv_heads, s.head_dim)))
    vp = O.bf16_round(rng.standard_normal((L, s.n_kv_heads, s.head_dim)))
    cos, sin = O.rope_cos_sin(st["pos"][0], s.head_dim, s.rope_theta)
    store = O.storer(s.dtype)
    t0 = time.perf_counter()
    O.layer_forward(s, lw, x, cos, sin, kp, vp, store)
    t_layer = time.perf_counter() - t0
    t0 = time.perf_counter()
    h = store(O.rmsnorm(x[:2], norm, s.rms_eps))
    O.softmax_scores(O.lm_head_logits(h, lm, s.mask_id))
    t_head2 = time.perf_counter() - t0
    t0 = time.perf_counter()
    H = rng.uniform(10, 12, W)
    O.select_eq11(H, st["pos"][0], st["obs"][0], wl.alpha, wl.tau)
    O.commit_run(st["obs"][0], st["pos"][0], L)
    t_sel = time.perf_counter() - t0
    B = wl.batch
    t_sample = t_layer + t_head2 + t_sel
    t_step = B * (s.n_layers * t_layer + (W / 2.0) * t_head2 + t_sel)
    hi = host_info()
    return {"value": ctx_commits_per_step / t_step, "unit": "committed tokens/s",
            "cores": hi["blas_threads"] or hi["cores"], "kind": "oracle",
            "sample": (f"extrapolated: 1 of {s.n_layers} layers x 1 of {B} sequences ({W} rows, "
                       f"prefix {L}), LM head on 2 of {B * W} rows and the selection of 1 "
                       f"sequence ran in {t_sample:.2f} s, scaled by the layers, sequences "
                       f"and rows of a whole step to {t_step:.1f} s"),
            "cpu": hi["cpu"], "host_cores": hi["cores"], "blas_threads": hi["blas_threads"],
            "seconds_per_step": t_step, "seconds_per_sample": t_sample}


def kernel_rates(tim, byts, hbm, n_steps, flops=None, tc=None):
    """Per-kind CUDA-event times of an eager pass -> launches, us per launch,
    algorithmic GB/s and fraction of the measured HBM bandwidth, and (with
    flops and the tensor peak tc in TFLOP/s) algorithmic TFLOP/s, fraction
    of the tensor peak and which of the two bounds the kind: the larger of
    bytes / HBM and FLOPs / tensor peak."""
    kernels = {}
    for kind, (kms, n) in tim.items():
        if n == 0:
            continue
        d = {"ms_total": round(kms, 4), "launches": n, "us_per_launch": round(1e3 * kms / n, 2),
             "launches_per_step": round(n / n_steps, 2)}
        t = kms / n * 1e-3
        if kind in byts:
            d["gbs"] = round(byts[kind] / t / 1e9, 1)
            d["frac_hbm"] = round(d["gbs"] / hbm, 3)
        if flops and tc and kind in flops:
            d["tflops"] = round(flops[kind] / t / 1e12, 1)
            d["frac_tensor"] = round(d["tflops"] / tc, 3)
            if kind in byts:
                d["bound"] = ("tensor" if flops[kind] / (tc * 1e12) > byts[kind] / (hbm * 1e9)
                              else "hbm")
        kernels[kind] = d
    return kernels


def measure(name, args, device, rank, world, weights=None, timed_steps=None, e2e=True,
            clocks=False, loop_steps=0):
    """Time one workload: the graph-replayed step loop (value), the same loop
    end to end through the Python API with host buffers (e2e), an eager
    pass with a CUDA-event pair around every launch (per-kernel rates,
    roofline) and, with loop_steps, the streaming loop run on the device
    (one wedlm_generate call: a conditional while node over the step).
    Returns (result dict, workload, state, weights, committed tokens per
    step)."""
    import torch
    from serving_wedlm_step_gb300 import binding as Bd
    from serving_wedlm_step_gb300.binding import WedlmContext
    steps = timed_steps or args.steps
    wl, st, w, pools, plant = setup(name, steps, args.warmup, device, weights, loop_steps)
    s = wl.shape
    B, W = wl.batch, wl.window
    ctx = WedlmContext(s, w, window=W, max_batch=B, max_pages_per_seq=st["max_pages"])
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    bufs = [{"tokens": T(st["tokens"]), "pos": T(st["pos"]), "obs": T(st["obs"])},
            {"tokens": T(st["tokens"]), "pos": T(st["pos"]), "obs": T(st["obs"])}]
    outs = [ctx.make_outputs(B, device=device), ctx.make_outputs(B, device=device)]
    for i in range(2):  # step i reads bufs[i], writes outs[i] = views of bufs[1-i]
        outs[i]["new_tokens"] = bufs[1 - i]["tokens"]
        outs[i]["new_pos"] = bufs[1 - i]["pos"]
        outs[i]["new_observed"] = bufs[1 - i]["obs"]
    seq_len = T(st["seq_len"])
    page_table = T(st["page_table"])
    plant_t = T(plant) if plant is not None else None
    bias = plant_bias_for(s.vocab) if plant is not None else 0.0
    stream = torch.cuda.current_stream(device)
    masked_rows = []

    def one(i, count_masked=False):
        b = bufs[i % 2]
        if count_masked:
            masked_rows.append(b["obs"].numel() - int(b["obs"].sum()))
        ctx.step(b["tokens"], b["pos"], b["obs"], seq_len, page_table, pools, st["num_pages"],
                 wl.alpha, wl.tau, outs[i % 2], plant_token=plant_t, plant_bias=bias,
                 stream=stream)

    k = 0
    for _ in range(args.warmup):
        one(k)
        k += 1
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError(f"{name}: device error word set during warm-up")
    len0 = int(seq_len.sum())
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if clocks else None
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one(k)
        k += 1
    e1.record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop() if sampler else None
    ms = e0.elapsed_time(e1)
    committed = int(seq_len.sum()) - len0
    ms, committed = reduce_over_ranks(ms, committed, world, device)
    if ctx.status() != 0:
        raise RuntimeError(f"{name}: device error word set during the timed steps")
    value = committed / (ms / 1e3)

    # ---- end to end through the Python API with host buffers -------------
    e2e_rec = None
    if e2e:
        e2e_steps = max(4, min(steps, 32))
        last = bufs[k % 2]
        # the window goes in as one pinned byte buffer (int32 tokens | int32
        # pos | uint8 observed) and the results come back as one (the packed
        # step outputs): one copy each way per step
        n = B * W
        in_bytes = 8 * n + n

        def window_views(buf):
            return {"tokens": buf[0:4 * n].view(torch.int32).view(B, W),
                    "pos": buf[4 * n:8 * n].view(torch.int32).view(B, W),
                    "obs": buf[8 * n:9 * n].view(B, W)}

        host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        host = window_views(host_in)
        for k2 in host:
            host[k2].copy_(last[k2].cpu())
        dev_in = torch.empty(in_bytes, dtype=torch.uint8, device=device)
        cur = window_views(dev_in)
        out = ctx.make_outputs(B, device=device, packed=True)
        host_out = torch.empty(out["packed"].numel(), dtype=torch.uint8).pin_memory()
        back = Bd.step_result_views(host_out, B, W)
        # NumPy views of the pinned buffers: the host side of a step (the
        # commit count, the next window) without a torch dispatch per op
        host_np = {k2: v.numpy() for k2, v in host.items()}
        back_np = {k2: v.numpy() for k2, v in back.items()}
        h2d, d2h = in_bytes, host_out.numel()
        n_e2e = 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            dev_in.copy_(host_in, non_blocking=True)
            ctx.step(cur["tokens"], cur["pos"], cur["obs"], seq_len, page_table, pools,
                     st["num_pages"], wl.alpha, wl.tau, out, plant_token=plant_t,
                     plant_bias=bias, stream=stream)
            host_out.copy_(out["packed"], non_blocking=True)
            stream.synchronize()
            n_e2e += int(back_np["n_committed"].sum())
            host_np["tokens"][...] = back_np["new_tokens"]
            host_np["pos"][...] = back_np["new_pos"]
            host_np["obs"][...] = back_np["new_observed"]
        e2e_s = time.perf_counter() - t0
        # committed tokens per step depend on where the sequences are, so the
        # step time is given too, for a like-for-like latency comparison
        e2e_rec = {"value": round(n_e2e / e2e_s, 2), "unit": "committed tokens/s",
                   "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                   "steps": e2e_steps, "ms_per_step": round(1e3 * e2e_s / e2e_steps, 4)}
        # continue from the state the end-to-end loop left
        for k2 in ("tokens", "pos", "obs"):
            bufs[k % 2][k2].copy_(host[k2].to(device))

    # ---- per-kernel CUDA-event timing (eager launches) --------------------
    ctx.set_timing(True)
    n_timing = 8
    for _ in range(n_timing):
        one(k, count_masked=True)
        k += 1
    torch.cuda.synchronize()
    tim = ctx.timings()
    ctx.set_timing(False)
    prefix_total = int(seq_len.sum()) - B * W  # lengths mid-run
    byts = algorithmic_bytes(s, B, W, prefix_total)
    n_masked = float(np.mean(masked_rows)) if masked_rows else float(B * W)
    flops = algorithmic_flops(s, B, W, prefix_total, n_masked)
    hbm, tc, peak_src = load_peaks()
    tc_sus, _ = load_tc_sustained()
    kernels = kernel_rates(tim, byts, hbm, n_timing, flops, tc)
    dom = max((k2 for k2 in kernels if k2 in byts), key=lambda k2: kernels[k2]["ms_total"])
    dk = kernels[dom]
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        traffic = json.load(open(tfile)).get(f"{name}:{dom}")
    if dk.get("bound") == "tensor":
        roofline = {"bound": "tensor", "kernel": dom, "achieved": dk["tflops"], "peak": tc,
                    "unit": "TFLOP/s", "frac": round(dk["tflops"] / tc, 3), "traffic": traffic,
                    "peak_source": f"{peak_src} bf16_tflops (cuBLAS burst)",
                    "algorithmic_flops_per_launch": flops[dom],
                    "algorithmic_bytes_per_launch": byts[dom]}
    else:
        roofline = {"bound": "hbm", "kernel": dom, "achieved": dk["gbs"], "peak": hbm,
                    "unit": "GB/s", "frac": round(dk["gbs"] / hbm, 3), "traffic": traffic,
                    "peak_source": f"{peak_src} hbm_gbs (copy)",
                    "algorithmic_bytes_per_launch": byts[dom]}
    # the whole step against its roofline: every kind at the larger of its
    # algorithmic bytes at the measured copy bandwidth and its FLOPs at the
    # sustained tensor peak, times its launches per step
    kind_launches = {k2: kernels[k2]["launches"] / n_timing for k2 in kernels if k2 in byts}
    step_bytes = sum(byts[k2] * n for k2, n in kind_launches.items())
    step_flops = sum(flops[k2] * n for k2, n in kind_launches.items())
    t_roof_ms = sum(max(byts[k2] / (hbm * 1e9), flops[k2] / (tc_sus * 1e12)) * n
                    for k2, n in kind_launches.items()) * 1e3
    step_roofline = {"bound": "per kind, the larger of hbm and tensor",
                     "algorithmic_bytes": int(step_bytes), "algorithmic_flops": int(step_flops),
                     "t_roof_ms": round(t_roof_ms, 4), "peak": hbm, "unit": "GB/s",
                     "tensor_peak": tc_sus, "tensor_unit": "TFLOP/s (sustained)",
                     "frac": round(t_roof_ms / (ms / steps), 3)}
    launches = ctx.launches_per_step(B)
    # ---- the streaming loop on the device ---------------------------------
    loop_rec = None
    if loop_steps:
        b = bufs[k % 2]
        done = torch.zeros(B, dtype=torch.int32, device=device)
        ran = torch.zeros(1, dtype=torch.int32, device=device)

        def loop(n):
            ctx.generate(b["tokens"], b["pos"], b["obs"], seq_len, page_table, pools,
                         st["num_pages"], wl.alpha, wl.tau, n, done, plant_token=plant_t,
                         plant_bias=bias, steps_run=ran, stream=stream)

        loop(2)  # builds and warms the loop graph
        torch.cuda.synchronize()
        l0 = int(seq_len.sum())
        e0.record(stream)
        loop(loop_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        if ctx.status() != 0:
            raise RuntimeError(f"{name}: device error word set in the device loop")
        lms = e0.elapsed_time(e1)
        n_run = int(ran.cpu()[0])
        lc = int(seq_len.sum()) - l0
        loop_rec = {"steps": n_run, "ms_per_step": round(lms / max(1, n_run), 4),
                    "value": round(lc / (lms / 1e3), 2), "unit": "committed tokens/s",
                    "committed": lc, "launches": "one graph launch (conditional while node)"}
    l2_note = (f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB moved per step)"
               if step_bytes > 129e6 else
               f"inputs smaller than L2 ({step_bytes / 1e6:.1f} MB per step, L2-resident)")
    per_step = committed / steps / world
    res = {
        "metric": "committed tokens/s of the window decode step (step latency in ms_per_step)",
        "value": round(value, 2), "unit": "committed tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(ms / steps, 4),
        "step_latency_us": round(1e3 * ms / steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if s.dtype == "bf16" else "f32",
        "data": "synthetic (seeded random-init weights N(0,0.02), random prefix KV N(0,1))",
        "config": {"workload": wl.describe(), "global_batch": B * world, "window": W,
                   "prefix": wl.prefix, "layers": s.n_layers, "alpha": wl.alpha,
                   "tau": wl.tau, "l2": l2_note, "planted_bias": bool(plant is not None),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        # committed tokens per forward per sequence, and the prefix cacheability
        # P_c = committed / processed token instances (Key claims §3.1, Eq. 4)
        "tokens_per_forward": round(per_step / B, 3),
        "committed_per_step": round(per_step, 3),
        "prefix_cacheability_Pc": round(per_step / (B * W), 4),
        "masked_rows_per_step": round(float(np.mean(masked_rows)), 1) if masked_rows else None,
        "gpu_launches": launches * steps,
        "launches_per_step": launches,
        "roofline": roofline,
        "step_roofline": step_roofline,
        "kernels": kernels,
    }
    if e2e_rec:
        res["e2e"] = e2e_rec
    if loop_rec:
        res["device_loop"] = loop_rec
    if clk:
        res["clocks"] = clk
    ctx.close()
    del pools
    return res, wl, st, w, per_step


def dual_stream_flops(n, block, nq, hd):
    """Algorithmic FLOPs of Dual-Stream attention: 4*hd per (query head,
    visible key) pair (QK^T and PV); memory row r sees r+1 keys, prediction
    row i (block j, physical index p) sees j*block + p + 1."""
    nb = n // block
    mem = n * (n + 1) // 2
    pred = block * block * nb * (nb - 1) // 2 + nb * block * (block + 1) // 2
    return 4 * hd * nq * (mem + pred)


def measure_dual_stream(device, n=4096, block=32, iters=10):
    """Time the Dual-Stream Masking attention (training-time memory and
    prediction streams) at the Qwen3-8B head shape: n tokens per stream,
    blocks of `block`.  Compute-bound: reported against the bf16 tensor
    peak."""
    import torch
    from serving_wedlm_step_gb300.binding import WedlmContext
    from synth import make_weights_torch, qwen3_layers
    s = qwen3_layers(1).replace(vocab=1024)
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    w = make_weights_torch(s, seed=0, device=device)
    # 512 workspace rows: partials for 2n/block blocks x 8 kv heads
    ctx = WedlmContext(s, w, window=1, max_batch=512, max_pages_per_seq=4)
    g = torch.Generator(device=device)
    g.manual_seed(0)
    q = torch.randn(2 * n, nq, hd, generator=g, device=device).to(torch.bfloat16)
    pool = torch.randn(n * 2 * nkv * hd, generator=g, device=device).to(torch.bfloat16)
    win = torch.randn(2 * n * 2 * nkv * hd, generator=g, device=device).to(torch.bfloat16)
    o = torch.empty(2 * n, nq * hd, dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(3):
        ctx.dual_stream_attention(n, block, q, pool, win, o, stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        ctx.dual_stream_attention(n, block, q, pool, win, o, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if ctx.status() != 0:
        raise RuntimeError("dual-stream attention: device error word set")
    ms = e0.elapsed_time(e1) / iters
    flops = dual_stream_flops(n, block, nq, hd)
    _, tf, src = load_peaks()
    achieved = flops / (ms * 1e-3) / 1e12
    ctx.close()
    return {"n": n, "block": block, "ms_per_call": round(ms, 4), "calls": iters,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": tf,
                         "unit": "TFLOP/s", "frac": round(achieved / tf, 3),
                         "algorithmic_flops": flops,
                         "peak_source": f"{src} bf16_tflops (cuBLAS burst)"}}


def measure_sweep(device, steps=32, alphas=(0.0, 0.01, 0.05), taus=(1.0, 2.0, 3.0)):
    """The quality/speed knob of Eq. 11 (Results: the distance penalty "set
    to balance quality and speed"): for each (alpha, tau), the streaming
    loop on the device from the same all-masked window over the two-layer
    low-entropy stack (prefix 32768, W = 32, batch 8, planted counting
    bias), reporting tokens committed per forward per sequence, slots filled
    per forward per sequence, and P_c (Key claims §3.1, Eq. 4)."""
    import torch
    from serving_wedlm_step_gb300.binding import WedlmContext
    wl, st, w, pools, plant = setup("two_layer_long", steps, 0, device)
    s = wl.shape
    B, W = wl.batch, wl.window
    ctx = WedlmContext(s, w, window=W, max_batch=B, max_pages_per_seq=st["max_pages"])
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    page_table = T(st["page_table"])
    plant_t = T(plant)
    bias = plant_bias_for(s.vocab)
    out = []
    for a in alphas:
        for t in taus:
            tok, pos, obs = T(st["tokens"]), T(st["pos"]), T(st["obs"])
            seq_len = T(st["seq_len"])
            done = torch.zeros(B, dtype=torch.int32, device=device)
            ran = torch.zeros(1, dtype=torch.int32, device=device)
            ctx.generate(tok, pos, obs, seq_len, page_table, pools, st["num_pages"], a, t,
                         steps, done, plant_token=plant_t, plant_bias=bias, steps_run=ran)
            torch.cuda.synchronize()
            if ctx.status() != 0:
                raise RuntimeError("sweep: device error word set")
            n = int(ran.cpu()[0])
            committed = int(seq_len.sum()) - int(np.asarray(st["seq_len"]).sum())
            filled = committed + int(obs.sum()) - int(np.asarray(st["obs"]).sum())
            out.append({"alpha": a, "tau": t, "steps": n,
                        "tokens_per_forward": round(committed / (n * B), 3),
                        "filled_per_forward": round(filled / (n * B), 3),
                        "prefix_cacheability_Pc": round(committed / (n * B * W), 4)})
    ctx.close()
    return {"workload": wl.describe(), "steps_per_point": steps, "points": out}


def run_ours(args):
    import torch
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    res, wl, st, w, per_step = measure(args.workload, args, device, rank, world, clocks=True)
    if rank == 0 and not args.no_cpu_baseline:
        cb = cpu_sample(wl, w, st, per_step)
        cb.pop("seconds_per_step", None)
        cb.pop("seconds_per_sample", None)
        res["cpu_baseline"] = cb
    extras = [e for e in extras_all(args) if e != args.workload and e in WORKLOADS]
    if extras_all(args):
        res["extra"] = {}
        for name in extras:
            # the full-stack workload shares the headline's weights (same
            # shape and seed); the others draw their own
            shared = w if WORKLOADS[name].shape == wl.shape and WORKLOADS[name].seed == wl.seed \
                else None
            torch.cuda.empty_cache()
            # the full stack runs the 256-step streaming loop both ways:
            # graph replays from the host and the loop on the device
            steps = 256 if name == "full_stack" else min(args.steps, 64)
            r, _, _, _, _ = measure(name, args, device, rank, world, weights=shared,
                                    timed_steps=steps, e2e=False,
                                    loop_steps=256 if name == "full_stack" else 0)
            keep = ("value", "unit", "steps", "ms_per_step", "step_latency_us",
                    "tokens_per_forward", "committed_per_step", "prefix_cacheability_Pc",
                    "masked_rows_per_step", "launches_per_step", "roofline", "step_roofline",
                    "kernels", "config", "device_loop")
            res["extra"][name] = {k: r[k] for k in keep if k in r}
        if "dual_stream" in extras_all(args):
            torch.cuda.empty_cache()
            res["extra"]["dual_stream"] = measure_dual_stream(device)
        if "sweep" in extras_all(args):
            torch.cuda.empty_cache()
            res["extra"]["alpha_tau_sweep"] = measure_sweep(device)
    if rank == 0:
        print(json.dumps(res))


def run_reference(args):
    """The oracle as it stands, on the host cores, each step a bounded
    sample of the same workload (see cpu_sample), on rank 0 only.  Each
    sample is one layer of one sequence plus two LM-head rows; the step time
    reported is extrapolated from it, and the line says so."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    from synth import make_weights_torch
    wl = WORKLOADS[args.workload]
    s = wl.shape
    st = make_state_np(wl)
    # the oracle needs one layer + the LM head: draw them on the CPU
    w = make_weights_torch(s.replace(n_layers=1), seed=wl.seed, device="cpu")
    # committed tokens per step: one per sequence, the least a step of the
    # stream commits on average (every step fills at least one slot of each
    # sequence).  The sample does not run the whole LM head, so it cannot
    # count the commits; the GPU arm counts its own (several per sequence on
    # the planted workload, and its cpu_baseline uses that count), so this
    # rate is a lower bound of the oracle's
    commits_per_step = float(wl.batch)
    samples, sample_s = [], []
    t_all = time.perf_counter()
    r = None
    for i in range(args.warmup + args.steps):
        r = cpu_sample(wl, w, st, commits_per_step)
        if i >= args.warmup:
            samples.append(r["seconds_per_step"])
            sample_s.append(r["seconds_per_sample"])
        if time.perf_counter() - t_all > 240:
            break
    t_step = statistics.median(samples) if samples else r["seconds_per_step"]
    value = commits_per_step / t_step
    res = {"impl": "reference",
           "metric": "committed tokens/s of the window decode step (step latency in ms_per_step)",
           "value": round(value, 6), "unit": "committed tokens/s", "n_gpus": world,
           "steps": len(samples), "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 1),
           "extrapolated": True, "commits_per_step_assumed": commits_per_step,
           "sample_seconds": round(statistics.median(sample_s), 3) if sample_s else None,
           "note": ("each of the `steps` samples runs one layer of one sequence, two LM-head "
                    "rows and one selection of the oracle; ms_per_step is that sample scaled "
                    "to a whole step, not a timed whole step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64", "data": "synthetic", "config": {"workload": wl.describe()},
           "cpu_baseline": {"value": round(value, 6), "unit": "committed tokens/s",
                            "cores": r["cores"], "kind": "oracle", "sample": r["sample"],
                            "cpu": r["cpu"], "blas_threads": r["blas_threads"]},
           "e2e": {"value": round(value, 6), "unit": "committed tokens/s",
                   "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

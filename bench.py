#!/usr/bin/env python3
"""Throughput of the TTT-E2E test-time inner loop (prefill) on one B300.

A step is one full pass of the inner loop over one synthetic sequence: reset
the context (initial fast weights, empty key/value ring), then ttt_prefill over
T tokens, i.e. for every chunk of b tokens the forward pass, the next-token
cross-entropy, the backward into the fast MLPs and their SGD step.  The
default workload is the 3B-class model at T = 131072 (window 8192, chunk 1024,
the MLPs of the last 7 of 28 blocks are fast), with seeded N(0, 0.02) weights
rounded to bf16 and Zipf(1.1) token ids.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is tokens/s over all ranks with the
inputs already resident on the device; `e2e` repeats the measurement through
the same C call with host (pinned) token and loss buffers, so the copies are
inside the timed region.  With N > 1 (torchrun) every rank runs its own
sequence (independent replicas: the chunk loop of one sequence is a strict
dependency chain and there is nothing to exchange).

`--impl reference` times the plain CPU oracle on the host cores on a bounded
sample of the same workload (the only other implementation of this method).

`--mode decode` measures decode-time test-time training instead: after an
untimed prefill of `--context` tokens, ttt_decode generates `--decode-tokens`
tokens greedily (one position per step, a test-time step on every completed
chunk); a step of the benchmark is one such decode call.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from long_context_lm_ttt_b300 import inputs  # noqa: E402

METRIC = "TTT-E2E prefill tokens/s at 3B, 128K ctx on 1 B300; % of dense BF16 peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
# kernel class, from one ncu capture of that class at the bench's shapes.  It
# is reported only while the sources the kernels are built from still hash to
# the value recorded with the capture; after any change it reads null until
# the capture is taken again.
TRAFFIC = {
    "gemm_fwd_bulk": {"bytes_per_launch": 642.4e6 + 185.8e6, "sha16": "8ef0b5979a31d5f5",
                      "sources": ("gemm_tc.cu", "common.cuh", "tc_common.cuh"),
                      "capture": "profiles/gemm_bulk_traffic_3b_T16384.md"},
}


def _sources_sha16(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "long_context_lm_ttt_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_of(kernel: str):
    t = TRAFFIC.get(kernel)
    if t is None:
        return None, None
    try:
        if _sources_sha16(t["sources"]) != t["sha16"]:
            return None, f"{t['capture']} (stale: the kernel sources changed since the capture)"
    except OSError:
        return None, None
    return t["bytes_per_launch"], t["capture"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="3b", choices=sorted(inputs.SHAPES))
    ap.add_argument("--T", type=int, default=None, help="sequence length (default: the config's)")
    ap.add_argument("--lr", type=float, default=None, help="override the SGD step (0: plain SWA forward)")
    ap.add_argument("--window", type=int, default=None,
                    help="override the attention window (>= T: full attention)")
    ap.add_argument("--fast-layers", type=int, default=None,
                    help="override the number of fast blocks (0: no test-time training, forward only)")
    ap.add_argument("--cpu-tokens", type=int, default=None,
                    help="tokens the oracle is timed on (default: one chunk from 760M up, four below; "
                         "--impl reference: 128 at 3B)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dual-mlp", action="store_true",
                    help="fast blocks carry a static second MLP after the fast one")
    ap.add_argument("--fast-bf16-single", action="store_true",
                    help="the forward reads the fast weights as one bf16 copy (default: the bf16 pair hi + lo)")
    ap.add_argument("--bulk-tokens", type=int, default=0,
                    help="tokens per super-chunk of the frozen blocks' bulk pass (0: automatic)")
    ap.add_argument("--mode", choices=["prefill", "decode", "batch"], default="prefill")
    ap.add_argument("--sequences", type=int, default=2,
                    help="batch: sequences read at once")
    ap.add_argument("--batch-impl", choices=["grouped", "contexts"], default="grouped",
                    help="batch: one context holding the sequences (stacked static products, grouped "
                         "fast-weight GEMMs), or one context per sequence run concurrently (ttt_prefill_batch)")
    ap.add_argument("--context", type=int, default=None,
                    help="decode: tokens prefilled before decoding (default 8 chunks)")
    ap.add_argument("--decode-tokens", type=int, default=None,
                    help="decode: tokens generated per step (default one chunk)")
    ap.add_argument("--profile", choices=["timed", "off"], default="timed",
                    help="per-launch CUDA events over a second, profiled pass of the timed steps (roofline), or none")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    rows.append((float(p[1]), float(p[2]), float(p[3]), p[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        pmax = max(r[2] for r in rows)
        load = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        reasons = sorted({self.REASONS[i] for r in load for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": pmax}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def workload(args, rank=0):
    s = inputs.shape(args.config)
    if args.T is not None:
        s = s.replace(seq_len=args.T)
    if args.lr is not None:
        s = s.replace(lr=args.lr)
    if args.window is not None:
        s = s.replace(window=args.window)
    if args.fast_layers is not None:
        s = s.replace(n_ttt_layers=args.fast_layers)
    if args.dual_mlp:
        s = s.replace(dual_mlp=True)
    tok = inputs.make_tokens(s, seed=1 + rank)
    return s, tok


def workload_name(s, args=None):
    single = bool(args is not None and getattr(args, "fast_bf16_single", False))
    return (f"{s.name} TTT-E2E prefill: L={s.n_layers} d={s.d_model} H={s.n_heads}/{s.n_kv_heads}x{s.head_dim} "
            f"ff={s.d_ff} V={s.vocab} W={s.window} b={s.chunk} T={s.seq_len} fast={s.n_ttt_layers} lr={s.lr}"
            + (" dual-MLP fast blocks" if s.dual_mlp else "")
            + (", fast weights fp32 master read as one bf16 copy" if single
               else ", fast weights fp32 master read as a bf16 hi+lo pair"))


def make_model(TT, s, w, args, max_tokens):
    return TT.TTT(s, w, TT.TTT_BF16, max_tokens=max_tokens, bulk_tokens=args.bulk_tokens,
                  fast_bf16_single=args.fast_bf16_single)


def cpu_baseline(s, w, tok, n_tokens):
    """The oracle as it stands, timed on the host cores over the first
    n_tokens positions (a prefix of the first chunk, or whole chunks).  Its
    state (an fp64 copy of every weight) is built before the timer starts;
    the timed region is the oracle's own chunk steps, in prefill's order."""
    from oracle import ttt_ref as O
    try:
        import psutil
        avail = psutil.virtual_memory().available
    except Exception:
        avail = 1 << 62
    dtype = np.float64 if avail > 3.2 * 8 * inputs.n_params(s) else np.float32
    cfg = O.OracleConfig.from_mapping(s.as_dict())
    sample = np.asarray(tok[:n_tokens])
    bounds = O.chunk_bounds(n_tokens, s.chunk)
    t0 = time.perf_counter()
    st = O.OracleState(cfg, w, max_positions=bounds[-1][1], dtype=dtype)
    setup = time.perf_counter() - t0
    t0 = time.perf_counter()
    for a, b in bounds:
        O.step_chunk(st, sample, a, b, cfg.lr)
    dt = time.perf_counter() - t0
    del st
    return {"value": n_tokens / dt, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"first {n_tokens} tokens of the sequence ({len(bounds)} chunk(s) of the {s.name} workload, "
                      f"same weights and ids), {np.dtype(dtype).name} numpy, {dt:.1f} s of chunk steps; the "
                      f"oracle's state set-up ({setup:.1f} s, a {np.dtype(dtype).name} copy of every weight) "
                      f"is outside the timed region"}


def default_cpu_tokens(s):
    # one whole chunk from the 760M class up (the 3B chunk is 1024 tokens),
    # four chunks below
    return s.chunk if s.d_model >= 1536 else min(s.seq_len, 4 * s.chunk)


def reference_tokens(s):
    # --impl reference repeats the sample warmup + steps times: a shorter
    # prefix of the first chunk at the largest shapes keeps the run to minutes
    return 128 if s.d_model >= 3072 else default_cpu_tokens(s)


# ---------------------------------------------------------------------------
def run_reference(args):
    """--impl reference: the CPU oracle, each step a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    s, tok = workload(args)
    w = inputs.make_weights(s)
    n = args.cpu_tokens or reference_tokens(s)
    times = []
    base = None
    for i in range(args.warmup + args.steps):
        b = cpu_baseline(s, w, tok, n)
        if i >= args.warmup:
            times.append(n / b["value"])
            base = b
    total = sum(times)
    v = n * args.steps / total
    base["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_name(s, args), "global_batch": 1,
                                            "seq_len": s.seq_len, "sample_tokens": n},
            "cpu_baseline": base,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def job_rate(local_ms: float, world: int, tokens_per_rank: int, steps: int, dist=None, device=None):
    """Whole-job throughput of independent replicas: every rank processed
    `steps` sequences of `tokens_per_rank` tokens; the job took as long as
    its slowest rank.  Returns (max_ms over ranks, tokens/s of the job)."""
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if dist is not None and world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, world * tokens_per_rank * steps / (ms_max / 1e3)


def roofline(prof, peaks, peak_src):
    dom = max(prof.items(), key=lambda kv: kv[1]["ms"])
    name, st = dom
    if st["launches"] == 0 or st["ms"] <= 0:
        return None, dom
    sec = st["ms"] / 1e3
    if st["flops"] > 0:
        ach = st["flops"] / sec / 1e12
        pk = peaks["bf16_tflops_sustained"]
        r = {"bound": "tensor", "achieved": ach, "peak": pk, "unit": "TFLOP/s", "frac": ach / pk}
    else:
        ach = st["bytes"] / sec / 1e9
        pk = peaks["hbm_gbs"]
        r = {"bound": "hbm", "achieved": ach, "peak": pk, "unit": "GB/s", "frac": ach / pk}
    traffic, src = traffic_of(name)
    r.update({"traffic": traffic, "kernel": name, "launches": st["launches"],
              "avg_launch_ms": st["ms"] / st["launches"],
              "algorithmic_bytes_per_launch": st["bytes"] / st["launches"],
              "peak_source": f"{peak_src} ({'sustained bf16' if r['bound'] == 'tensor' else 'copy'})"})
    if src:
        r["traffic_source"] = src
    return r, dom


def run_ours(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from long_context_lm_ttt_b300 import ttt as TT
    TT.load()
    peaks, peak_src = load_peaks()

    s, tok = workload(args, rank)
    T = s.seq_len
    nC = s.n_chunks
    t_setup = time.perf_counter()
    w = inputs.make_weights(s)
    m = make_model(TT, s, w, args, T)
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if not want_cpu:
        del w
    t_setup = time.perf_counter() - t_setup

    tok_d = torch.from_numpy(tok).cuda()
    loss_d = torch.zeros(nC, dtype=torch.float32, device="cuda")

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def step(tk, ls):
        m.reset()
        m.prefill(tk, ls)

    for _ in range(args.warmup):
        step(tok_d, loss_d)
    losses = loss_d.cpu().numpy()
    if not np.all(np.isfinite(losses)):
        raise SystemExit(f"non-finite chunk losses: {losses}")

    uuid = str(torch.cuda.get_device_properties(local).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    barrier()
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        step(tok_d, loss_d)
    ev1.record()
    barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms_max, value = job_rate(ms, world, T, args.steps, dist, device="cuda")

    # The same K steps again with per-launch events.  Profiling runs the bulk
    # pass and the chunk loop on one stream, so each event pair times one
    # kernel alone; this pass is slower than the timed one by the overlap.
    prof, prof_ms = None, None
    if args.profile == "timed":
        m.profile(True)
        barrier()
        ev0.record()
        for _ in range(args.steps):
            step(tok_d, loss_d)
        ev1.record()
        barrier()
        prof_ms = ev0.elapsed_time(ev1) / args.steps
        prof = m.profile_read()
        m.profile(False)

    # end to end through the same call with host buffers (pinned)
    e2e = None
    if not args.no_e2e:
        tok_h = torch.from_numpy(tok).pin_memory()
        loss_h = torch.zeros(nC, dtype=torch.float32).pin_memory()
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step(tok_h, loss_h)
        barrier()
        _, e2e_value = job_rate(1e3 * (time.perf_counter() - t0), world, T, args.steps, dist, device="cuda")
        e2e = {"value": e2e_value, "unit": UNIT,
               "h2d_bytes_per_step": int(tok_h.numel() * 4), "d2h_bytes_per_step": int(loss_h.numel() * 4)}

    fl = inputs.flops_per_sequence(s)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(s, args), "global_batch": world, "seq_len": T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (every chunk streams all weights, 6+ GB at 3B)"},
        "clocks": {"sm_mhz": clk.get("sm_mhz"), "sm_max_mhz": clk.get("sm_max_mhz"), "reasons": clk.get("reasons")},
        "e2e": e2e,
        "model_tflops": fl["total"] * world * args.steps / (ms_max / 1e3) / 1e12,
        "frac_of_peak": {"burst": fl["total"] * world * args.steps / (ms_max / 1e3) / 1e12 / peaks["bf16_tflops"],
                         "sustained": fl["total"] * world * args.steps / (ms_max / 1e3) / 1e12
                         / peaks["bf16_tflops_sustained"], "peaks": peak_src},
        "setup_s": t_setup,
    }
    if prof is not None:
        rl, _ = roofline(prof, peaks, peak_src)
        if rl is not None:
            rl["measured"] = "CUDA events around each launch, profiled pass of the same steps, one stream"
        line["roofline"] = rl
        line["profiled_ms_per_step"] = prof_ms
        line["gpu_launches"] = int(sum(v["launches"] for v in prof.values()))
        tot = sum(v["ms"] for v in prof.values()) or 1.0
        line["kernels"] = {k: {"launches": v["launches"], "ms_per_step": v["ms"] / args.steps,
                               "share": v["ms"] / tot,
                               "tflops": (v["flops"] / (v["ms"] / 1e3) / 1e12) if v["ms"] > 0 and v["flops"] else None,
                               "gbs": (v["bytes"] / (v["ms"] / 1e3) / 1e9) if v["ms"] > 0 else None}
                           for k, v in prof.items() if v["launches"]}
    if want_cpu:
        n = args.cpu_tokens or default_cpu_tokens(s)
        line["cpu_baseline"] = cpu_baseline(s, w, tok, n)
    m.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def decode_bytes_per_token(s, ctx: int) -> float:
    """HBM bytes one decode step must read: every weight once (the fast
    MLPs as the bf16 pair), the window's keys and values in every layer,
    and one embedding row."""
    d, ff, H, Hkv, hd, L, Lt = s.d_model, s.d_ff, s.n_heads, s.n_kv_heads, s.head_dim, s.n_layers, s.n_ttt_layers
    attn = d * (H + 2 * Hkv) * hd + H * hd * d
    mlp = 3 * d * ff
    w = 2.0 * (L * attn + (L - Lt) * mlp + 2 * Lt * mlp + s.vocab * d + d)
    kv = 2.0 * 2 * L * min(ctx, s.window) * Hkv * hd
    return w + kv


def run_decode(args):
    """--mode decode: tokens/s of one sequence generating greedily with a
    test-time step on every completed chunk."""
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and int(os.environ.get("RANK", "0")) != 0:
        return 0
    torch.cuda.set_device(0)
    from long_context_lm_ttt_b300 import ttt as TT
    TT.load()
    peaks, peak_src = load_peaks()
    s, tok = workload(args)
    b = s.chunk
    ctx = args.context if args.context is not None else 8 * b
    nd = args.decode_tokens or b
    if ctx % b:
        raise SystemExit("--context must be a multiple of the chunk length")
    w = inputs.make_weights(s)
    tok = inputs.make_tokens(s.replace(seq_len=ctx + 1), seed=1)
    m = make_model(TT, s, w, args, ctx + nd + 1)
    del w
    tok_d = torch.from_numpy(tok).cuda()
    out_d = torch.zeros(nd + 1, dtype=torch.int32, device="cuda")
    loss_d = torch.zeros(nd // b + 1, dtype=torch.float32, device="cuda")
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def step(host=False):
        m.reset()
        m.prefill(tok_d[:ctx])
        torch.cuda.synchronize()
        if host:
            t0 = time.perf_counter()
            o, l = m.decode(tok[ctx:ctx + 1], nd)
            return 1e3 * (time.perf_counter() - t0), o
        ev0.record()
        # an NVTX range, so that a profiler can take the decode launches alone
        torch.cuda.nvtx.range_push("decode")
        m.decode(tok_d[ctx:ctx + 1], nd, out_d, loss_d)
        torch.cuda.nvtx.range_pop()
        ev1.record()
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1), None

    for _ in range(args.warmup):
        step()
    uuid = str(torch.cuda.get_device_properties(0).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    clocks.start()
    ms = [step()[0] for _ in range(args.steps)]
    clk = clocks.stop()
    dec_ms = sum(ms)
    value = nd * args.steps / (dec_ms / 1e3)
    if not np.all(np.isfinite(loss_d.cpu().numpy()[: nd // b])):
        raise SystemExit("non-finite decode chunk loss")
    e2e_ms = sum(step(host=True)[0] for _ in range(args.steps))
    # one more decode call with per-launch events (classes as in the
    # prefill profile; the test-time step of the completed chunk included)
    kernels = None
    if args.profile == "timed":
        m.reset()
        m.prefill(tok_d[:ctx])
        torch.cuda.synchronize()
        m.profile(True)
        m.decode(tok_d[ctx:ctx + 1], nd, out_d, loss_d)
        prof = m.profile_read()
        m.profile(False)
        tot = sum(v["ms"] for v in prof.values()) or 1.0
        kernels = {k: {"launches": v["launches"], "ms_per_token": v["ms"] / nd, "share": v["ms"] / tot,
                       "gbs": (v["bytes"] / (v["ms"] / 1e3) / 1e9) if v["ms"] > 0 else None}
                   for k, v in prof.items() if v["launches"]}
    per_tok = dec_ms / args.steps / nd
    bytes_tok = decode_bytes_per_token(s, ctx + nd // 2)
    ach = bytes_tok / (per_tok / 1e3) / 1e9
    line = {
        "metric": "TTT-E2E decode-time test-time training, tokens/s of one sequence (greedy, "
                  "one test-time step per chunk of generated tokens)",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dec_ms / args.steps, "ms_per_token": per_tok, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(s, args) + f" decode: context {ctx}, {nd} generated tokens",
                   "global_batch": 1, "context": ctx, "decode_tokens": nd,
                   "l2": "every step streams all weights (7+ GB at 3B), larger than L2"},
        "clocks": {"sm_mhz": clk.get("sm_mhz"), "sm_max_mhz": clk.get("sm_max_mhz"), "reasons": clk.get("reasons")},
        "e2e": {"value": nd * args.steps / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4 * (nd + 1) + 4 * (nd // b + 1)},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "whole decode step (weights + window keys/values per token; the chunk "
                               "steps' time is included, their bytes are not)",
                     "peak_source": f"{peak_src} (copy)"},
    }
    if kernels is not None:
        line["kernels"] = kernels
        line["gpu_launches_per_token"] = sum(v["launches"] for v in kernels.values()) / nd
    m.close()
    print(json.dumps(line), flush=True)
    return 0


def run_batch(args):
    """--mode batch: tokens/s of B sequences read at once, each with its own
    fast weights.  grouped: one context with n_seq = B (one ttt_prefill; the
    products with static weights take every sequence's rows in one launch,
    the fast MLPs' products are grouped GEMMs).  contexts: B contexts run
    concurrently by ttt_prefill_batch, one stream each.  A step resets and
    prefills all B sequences."""
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and int(os.environ.get("RANK", "0")) != 0:
        return 0
    torch.cuda.set_device(0)
    from long_context_lm_ttt_b300 import ttt as TT
    TT.load()
    B = args.sequences
    s, _ = workload(args)
    T = s.seq_len
    w = inputs.make_weights(s)
    grouped = args.batch_impl == "grouped"
    if grouped:
        models = [TT.TTT(s, w, TT.TTT_BF16, max_tokens=T, bulk_tokens=args.bulk_tokens,
                         fast_bf16_single=args.fast_bf16_single, n_seq=B)]
    else:
        models = [make_model(TT, s, w, args, T) for _ in range(B)]
    del w
    toks = [torch.from_numpy(inputs.make_tokens(s, seed=1 + i)).cuda() for i in range(B)]
    if grouped:
        tok_all = torch.stack(toks).contiguous()
        loss_all = torch.zeros((B, s.n_chunks), dtype=torch.float32, device="cuda")
    losses = [torch.zeros(s.n_chunks, dtype=torch.float32, device="cuda") for _ in range(B)]
    streams = [torch.cuda.Stream() for _ in range(B)]
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def step():
        for m in models:
            m.reset()
        torch.cuda.synchronize()
        if grouped:
            ev0.record()
            models[0].prefill(tok_all, loss_all)
            ev1.record()
            torch.cuda.synchronize()
            return ev0.elapsed_time(ev1) / 1e3
        t0 = time.perf_counter()
        TT.ttt_prefill_batch([m.ctx for m in models], toks, [T] * B, losses, streams)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    if grouped and not torch.isfinite(loss_all).all():
        raise SystemExit("non-finite chunk losses")
    uuid = str(torch.cuda.get_device_properties(0).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    clocks.start()
    sec = sum(step() for _ in range(args.steps))
    clk = clocks.stop()
    value = B * T * args.steps / sec
    fl = inputs.flops_per_sequence(s)
    how = ("one context, stacked static products and grouped fast-weight GEMMs" if grouped
           else "concurrent contexts")
    line = {
        "metric": f"TTT-E2E prefill tokens/s, {B} sequences per call ({how})",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(s, args) + f", {B} sequences", "global_batch": B, "seq_len": T,
                   "batch_impl": args.batch_impl},
        "clocks": {"sm_mhz": clk.get("sm_mhz"), "sm_max_mhz": clk.get("sm_max_mhz"), "reasons": clk.get("reasons")},
        "model_tflops": fl["total"] * B * args.steps / sec / 1e12,
        "timing": ("CUDA events around each ttt_prefill" if grouped else
                   "host wall clock around each ttt_prefill_batch call (it returns after the work has completed)"),
    }
    for m in models:
        m.close()
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "decode":
        return run_decode(args)
    if args.mode == "batch":
        return run_batch(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

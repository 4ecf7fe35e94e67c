#!/usr/bin/env python
"""Benchmark of the fused GRPO selective-log-prob loss forward + backward.

One step = one grpo_loss_fwd_bwd call over one synthetic batch: the logit GEMM
with online log-sum-exp over the whole vocabulary, the loss / dlogp epilogue,
and the chunked backward (recomputed logit tiles -> G -> dH). Default workload:
the Llama-3.1-8B lm_head shape (N = 1 x 4 x 4096 tokens, D = 4096,
V = 128256, bf16), inputs resident in HBM and larger than L2 (W is 1.05 GB,
hidden 134 MB), so no L2 flush is needed between steps.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0). Under torchrun each rank runs its own
independent batch (weak scaling, no collective on the data path); the time is
the max over ranks.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s & % bf16 tensor peak, GRPO logp+loss fwd+bwd (Llama-3.1-8B shape)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama-3.1-8b")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override tokens per completion (small profiling cases)")
    ap.add_argument("--chunk-tokens", type=int, default=0)
    ap.add_argument("--vocab-block", type=int, default=0)
    ap.add_argument("--backward", default="auto",
                    choices=["auto", "stored", "single_pass", "recompute"],
                    help="auto: the library's default choice (flags 0) for the workspace "
                         "budget; stored: the backward reads fp16 logits kept per chunk "
                         "(4NDV executed); single_pass: one vocabulary block of logits at a "
                         "time, rescaled U accumulator (4NDV); recompute: it recomputes "
                         "the logit tiles (6NDV)")
    ap.add_argument("--workspace-limit-gb", type=float, default=0.0,
                    help="workspace budget passed to the library (0 = none)")
    ap.add_argument("--budget-sweep", default="",
                    help="no headline line: comma-separated workspace budgets in GB; for "
                         "each, time the automatic choice and both forced forms and print "
                         "one JSON line per (budget, form)")
    ap.add_argument("--single-cta", action="store_true",
                    help="one CTA per 128-row GEMM tile instead of CTA pairs")
    ap.add_argument("--with-dw", action="store_true",
                    help="also compute the lm_head gradient dW (full fine-tuning; +2NDV)")
    ap.add_argument("--no-variant", action="store_true",
                    help="skip timing the other backward forms")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="no benchmark: turn an ncu launch list (--csv, with "
                         "gpu__time_duration.sum, dram__bytes_read.sum and "
                         "dram__bytes_write.sum) of this bench's calls into "
                         "profiles/traffic_<workload>_<backward>.json")
    ap.add_argument("--record-command", default="",
                    help="the command that made --record-traffic's CSV (kept in the record)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- helpers ----

def rank_env():
    """(world size, rank, local rank) as torch.distributed.run sets them."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(seed, rank):
    """Each replica draws its own batch: the job's work grows with the ranks (weak scaling)."""
    return seed + rank


def max_over_ranks(x):
    """The job's time is its slowest rank's: max of a float over all ranks."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# grpo_params.flags of each backward form (GRPO_FLAG_STORED_LOGITS,
# GRPO_FLAG_SINGLE_PASS, GRPO_FLAG_RECOMPUTE_LOGITS; 0 lets the library choose).
FORM_FLAGS = {"auto": 0, "stored": 1, "single_pass": 32, "recompute": 16}
FORM_NAMES = {"stored": "stored fp16 logits", "single_pass": "single pass over vocab blocks",
              "recompute": "recomputed logits"}
# Executed tensor work per valid token in units of D V (without dW): the
# stored and single-pass forms compute each logit once, the recomputed form twice.
EXECUTED_NDV = {"stored": 4.0, "single_pass": 4.0, "recompute": 6.0}


def form_of(plan):
    """The backward form a plan (grpo_get_plan) uses."""
    if plan["stored_logits"]:
        return "stored"
    return "single_pass" if plan.get("single_pass") else "recompute"


def flops_per_token(D, V):
    # 2DV forward + 4DV backward (recomputed logits + G W), per valid token.
    return 6.0 * D * V


def oracle_rows_per_second(p, target_s, seed, cores_note, gpu=None, masked_loss=None):
    """Time the fp64 oracle on a seeded sample of valid rows of workload `p`.

    gpu = (old, ref, logp, dH) of a GPU call on the same inputs: the oracle
    then runs with that call's old/ref log-probs, and its rows are compared
    with the call's logp and dH (each row is exact given the loss
    denominator). masked_loss(mask) runs the same call with another mask and
    returns its loss: with the sampled rows as the mask, the oracle's loss
    over those rows is exact, so the loss is compared too. Returns (rows,
    seconds, parity dict or None)."""
    import numpy as np
    import torch

    import oracle

    rng = np.random.default_rng(seed)
    valid = torch.nonzero(p.mask.cpu() != 0).flatten().numpy()
    W64 = p.weight.float().cpu().numpy().astype(np.float64)  # input preparation
    h = p.hidden.cpu()
    ids = p.ids.cpu().numpy()
    if gpu is None:
        base = torch.full((p.n_tokens,), -math.log(p.vocab))
        old, ref = (x.cpu() for x in p.old_ref(base.to(p.old_noise.device)))
    else:
        old, ref = gpu[0].cpu(), gpu[1].cpu()
    adv = p.adv.cpu()
    M = float(len(valid))

    def run(n_rows):
        rows = np.sort(rng.choice(valid, size=min(n_rows, len(valid)), replace=False))
        t0 = time.perf_counter()
        out = oracle.rows_fwd_bwd(h, W64, ids, rows, old, ref, adv, p.seq_len, M,
                                  p.eps_low, p.eps_high, p.beta)
        return rows, time.perf_counter() - t0, out

    run(4)  # the first call pays one-time costs (thread pool start-up, page-in)
    rows0, t0, _ = run(24)
    per_row = t0 / len(rows0)
    n_rows = int(max(8, min(len(valid), target_s / max(per_row, 1e-6))))
    rows, t, want = run(n_rows)
    parity = None
    if gpu is not None:
        idx = torch.from_numpy(rows)
        got_lp = gpu[2].cpu().double()[idx].numpy()
        got_dh = gpu[3][idx.to(gpu[3].device)].double().cpu().numpy()
        parity = {
            "rows": len(rows),
            "max_abs_dlogp": float(np.abs(got_lp - want["logp"]).max()),
            "rel_fro_dH": float(np.linalg.norm(got_dh - want["dH"]) /
                                np.linalg.norm(want["dH"])),
            "gates": "|dlogp| <= 1e-2, rel loss <= 1e-3, rel dH <= 2e-2"}
        if masked_loss is not None:
            # Same call with only the sampled rows unmasked: its loss is the
            # masked mean over exactly the rows the oracle computed.
            mask2 = torch.zeros(p.n_tokens, dtype=torch.uint8)
            mask2[idx] = 1
            lp_full = np.zeros(p.n_tokens)
            lp_full[rows] = want["logp"]
            L_want = oracle.grpo_loss(lp_full, old, ref, adv, mask2, p.seq_len, p.eps_low,
                                      p.eps_high, p.beta)[0]
            L_got = masked_loss(mask2)
            parity.update({"loss_rows": len(rows), "loss": L_got, "loss_oracle": L_want,
                           "rel_loss": abs(L_got - L_want) / abs(L_want),
                           "loss_note": "second call, same inputs, mask = the sampled rows "
                                        "(the oracle's loss over them is exact)"})
    return len(rows), t, parity


def code_tokens(src):
    """C/C++/CUDA source without comments and with whitespace collapsed."""

    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # string or character literal, kept verbatim
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash():
    """Hash of the CUDA sources' code (comments and layout ignored): DRAM traffic
    recorded for other code is stale."""
    import hashlib

    csrc = os.path.join(ROOT, "chunked_log_prob_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_path(workload, backward):
    return os.path.join(ROOT, "profiles", f"traffic_{workload}_{backward}.json")


def recorded_traffic(workload, backward):
    """The committed ncu DRAM record of one call, if it matches these sources."""
    try:
        with open(traffic_path(workload, backward)) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec


_NCU_SCALE = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
              "ns": 1e-6, "nsecond": 1e-6, "us": 1e-3, "usecond": 1e-3, "ms": 1.0,
              "msecond": 1.0, "s": 1e3, "second": 1e3}
_FIRST_KERNEL = "row_plan_kernel"  # every grpo_loss_fwd_bwd call starts with it
# The library's kernels (any other launch in a capture is torch's own).
LIBRARY_KERNELS = ("tc_gemm_kernel", "finalize_kernel", "finalize_gform_kernel",
                   "finalize_rows_kernel", "single_pass_p_kernel", "finish_loss_kernel",
                   "row_plan_kernel", "zero_padding_blocks_kernel", "seq_lens_kernel",
                   "tail_fixup_kernel", "gather_blocks_kernel", "bounded_wait_selftest_kernel")


def ncu_launches(csv_path):
    """The library's launches in an ncu --csv capture, in launch order:
    {"name", "read", "write", "ms"} (bytes, milliseconds); launches of other
    code (torch's own kernels) are dropped."""
    import csv

    with open(csv_path, newline="") as f:
        rows = list(csv.reader(f))
    head = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    h = rows[head]
    col = {k: h.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Unit",
                                   "Metric Value")}
    launches = {}
    for r in rows[head + 1:]:
        if len(r) < len(h):
            continue
        d = launches.setdefault(int(r[col["ID"]]), {"name": r[col["Kernel Name"]]})
        d[r[col["Metric Name"]]] = (float(r[col["Metric Value"]].replace(",", ""))
                                    * _NCU_SCALE[r[col["Metric Unit"]]])
    seq = []
    for i in sorted(launches):
        d = launches[i]
        # ncu prints "void grpo::tc_gemm_kernel<(int)3, (int)2>(...)" or, with
        # other name bases, "void tc_gemm_kernel<3, 2>(...)".
        name = d["name"].replace("(int)", "").split("(")[0]
        name = name.replace("void ", "").replace("grpo::", "").strip()
        if name.split("<")[0] not in LIBRARY_KERNELS:
            continue
        seq.append({"name": name, "read": d.get("dram__bytes_read.sum", 0.0),
                    "write": d.get("dram__bytes_write.sum", 0.0),
                    "ms": d.get("gpu__time_duration.sum", 0.0)})
    return seq


def ncu_calls(csv_path):
    """Split an ncu --csv launch list into the library's calls: lists of
    launches as ncu_launches gives them. A call runs from one row_plan_kernel
    launch up to the next; the last call, which the capture limit may have cut
    short, is dropped."""
    seq = ncu_launches(csv_path)
    starts = [i for i, d in enumerate(seq) if d["name"] == _FIRST_KERNEL]
    return [seq[a:b] for a, b in zip(starts, starts[1:])]


def record_traffic(csv_path, workload, backward, command):
    """Write the DRAM record of an ncu capture: of the last complete call in a
    launch list, or, when the capture holds no whole call (one kernel, a few
    launches, -k/-c; several such captures may be given, comma-separated), of
    each captured kernel per launch. The bench reads the dominant kernel's
    bytes per launch from either."""
    paths = csv_path.split(",")
    calls = ncu_calls(paths[0]) if len(paths) == 1 else []
    if not calls:
        seq = [d for pth in paths for d in ncu_launches(pth)]
        if not seq:
            raise SystemExit(f"{csv_path}: no launch of the library")
        per = {}
        for d in seq:
            e = per.setdefault(d["name"], {"launches": 0, "read_bytes": 0.0,
                                           "write_bytes": 0.0, "time_ms": 0.0})
            e["launches"] += 1
            e["read_bytes"] += d["read"]
            e["write_bytes"] += d["write"]
            e["time_ms"] += d["ms"]
        rec = {"workload": workload, "backward": backward, "dram_bytes_per_call": None,
               "scope": "captured launches of single kernels (no whole call); per_kernel "
                        "sums over them", "per_kernel": per, "command": command,
               "kernel_source_hash": kernel_source_hash()}
        with open(traffic_path(workload, backward), "w") as f:
            json.dump(rec, f, indent=1)
        return rec
    call = calls[-1]
    per = {}
    for d in call:
        e = per.setdefault(d["name"], {"launches": 0, "read_bytes": 0.0, "write_bytes": 0.0,
                                       "time_ms": 0.0})
        e["launches"] += 1
        e["read_bytes"] += d["read"]
        e["write_bytes"] += d["write"]
        e["time_ms"] += d["ms"]
    rd, wr = sum(d["read"] for d in call), sum(d["write"] for d in call)
    rec = {"workload": workload, "backward": backward, "dram_bytes_per_call": rd + wr,
           "dram_read_bytes": rd, "dram_write_bytes": wr, "launches_per_call": len(call),
           "ncu_time_ms_per_call": sum(d["ms"] for d in call), "per_kernel": per,
           "command": command, "kernel_source_hash": kernel_source_hash()}
    with open(traffic_path(workload, backward), "w") as f:
        json.dump(rec, f, indent=1)
    return rec


def kernel_work(name, D, V):
    """Algorithmic work of one kernel kind per valid token: (bound, amount, unit)."""
    if name.startswith("tc_gemm_kernel"):
        return "tensor", 2.0 * D * V, "flop"  # one pass of the N x V x D contraction
    if name in ("finalize_gform_kernel", "single_pass_p_kernel"):
        # fp16 logit row in, bf16 G (or P) row out, one fp32 maximum per 64-column
        # box: over a call, every vocabulary column of every valid token once
        return "hbm", 4.0 * V + 4.0 * math.ceil(V / 64), "byte"
    return None


def kernel_roofline(times, calls, D, V, valid, peaks, rec, call_ms=None):
    """Roofline of the kernel with the most device time over `calls` calls.

    times: per-kernel sums from the library's launch timing (CUDA events on
    each launch's own stream). A launch's algorithmic work is the kind's work
    per valid token x the valid tokens of a call / its launches per call.
    share: of the summed kernel time; of_call: of the call's own duration
    (kernels on the side stream overlap the others, so these may sum past 1)."""
    if not times:
        return None
    summed = sum(k["total_ms"] for k in times)
    per_kernel = [{"name": k["name"], "launches_per_call": k["launches"] / calls,
                   "avg_launch_ms": k["total_ms"] / k["launches"],
                   "ms_per_call": k["total_ms"] / calls,
                   "share": k["total_ms"] / summed,
                   "of_call": None if not call_ms else k["total_ms"] / calls / call_ms}
                  for k in sorted(times, key=lambda k: -k["total_ms"])]
    top = per_kernel[0]
    out = {"kernel": top["name"], "avg_launch_ms": top["avg_launch_ms"],
           "launches_per_call": top["launches_per_call"], "share": top["share"]}
    traffic = None
    if rec is not None and top["name"] in rec.get("per_kernel", {}):
        e = rec["per_kernel"][top["name"]]
        traffic = (e["read_bytes"] + e["write_bytes"]) / e["launches"]
    work = kernel_work(top["name"], D, V)
    if work is None:
        out.update({"bound": None, "achieved": None, "peak": None, "unit": None,
                    "frac": None, "traffic": traffic})
    else:
        bound, per_token, unit = work
        per_launch = per_token * valid / top["launches_per_call"]
        rate = per_launch / (top["avg_launch_ms"] / 1e3)
        if bound == "tensor":
            # The burst peak: a launch lasts milliseconds, not the seconds the
            # sustained figure's loop ran for; the sustained fraction beside it.
            achieved, peak, u = rate / 1e12, peaks["bf16_tflops"], "TFLOP/s"
            out["frac_of_sustained_peak"] = achieved / peaks["bf16_tflops_sustained"]
        else:
            achieved, peak, u = rate / 1e9, peaks["hbm_gbs"], "GB/s"
        out.update({"bound": bound, "achieved": achieved, "peak": peak, "unit": u,
                    "frac": achieved / peak, "traffic": traffic,
                    f"algorithmic_{unit}s_per_launch": per_launch})
    out["per_kernel"] = per_kernel
    return out


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- ours ----

def run_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as clp
    import synth

    over = {"T": args.seq_len} if args.seq_len > 0 else {}
    if args.seq_len > 0 and synth.WORKLOADS[args.workload]["lengths"] is not None:
        lo, hi = synth.WORKLOADS[args.workload]["lengths"]
        over["lengths"] = (min(lo, args.seq_len), args.seq_len)
    p = synth.make_problem(args.workload, seed=rank_seed(args.seed, rank), device=dev, **over)
    torch.cuda.empty_cache()  # drop the generator's fp32 temporaries
    N, D, V, T = p.n_tokens, p.hidden_size, p.vocab, p.seq_len
    limit = int(args.workspace_limit_gb * (1 << 30))

    def make(flag):
        return clp.make_params(p.eps_low, p.eps_high, p.beta, 0.0, args.chunk_tokens,
                               args.vocab_block, flags=flag | (2 if args.single_cta else 0),
                               workspace_limit_bytes=limit)

    params = make(FORM_FLAGS[args.backward])
    plan = clp.grpo_get_plan(N, D, V, T, params)
    stored = bool(plan["stored_logits"])
    form = form_of(plan)
    others = {f: make(FORM_FLAGS[f]) for f in ("stored", "single_pass", "recompute") if f != form}
    if args.backward == "auto":
        choice = ("library default (flags 0): the planner's automatic choice; %s; among the "
                  "forms that fit, %s has the shortest modelled GEMM time" % (
                      "no workspace budget" if limit == 0
                      else "budget %.2f GB" % args.workspace_limit_gb, FORM_NAMES[form]))
    else:
        choice = "forced by --backward %s" % args.backward
    ws_bytes = max(clp.grpo_workspace_size(N, D, V, T, params),
                   0 if args.no_variant else max(clp.grpo_workspace_size(N, D, V, T, o)
                                                 for o in others.values()))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    # old/ref: the policy's own log-probs (as a GRPO trainer gets them) + noise.
    base, _ = clp.grpo_logp_fwd(p.hidden, p.weight, p.ids, params=params, workspace=ws)
    old, ref = p.old_ref(base)
    valid = p.n_valid
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    dH = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, D, dtype=torch.float32, device=dev) if args.with_dw else None

    def step(prm=params):
        clp.grpo_loss_fwd_bwd(p.hidden, p.weight, p.ids, p.mask, old, ref, p.adv, T,
                              params=prm, workspace=ws, loss=loss, logp=logp, dH=dH, dW=dW)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    status = clp.grpo_read_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} ({clp.status_string(status)})")

    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = f"GPU-{gpu_id}" if gpu_id is not None else str(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Per-kernel device times over the timed calls: the library brackets each
    # launch with CUDA events on that launch's own stream (the caller's or its
    # side stream) and sums them per kernel (64K launches at most per read).
    launches_est = plan["launches_loss"] + (plan["n_chunks"] * plan["n_vocab_blocks"]
                                            if args.with_dw else 0)
    timed_calls = args.steps if args.steps * launches_est <= 60000 else 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_id) as clocks:
        time.sleep(0.3)  # let the sampler start
        clp.grpo_launch_timing_enable(timed_calls > 0)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        clp.grpo_launch_timing_enable(False)
    if world > 1:
        dist.barrier()
    ms_max = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    if timed_calls == 0:  # too many launches for one read: time 10 calls of their own
        timed_calls = 10
        clp.grpo_launch_timing_enable(True)
        for _ in range(timed_calls):
            step()
        torch.cuda.synchronize(dev)
        clp.grpo_launch_timing_enable(False)
    kernel_times = clp.grpo_launch_timing_read()

    # The other backward forms on the same inputs (reported beside the headline).
    variants = []
    if not args.no_variant:
        for f, prm in others.items():
            for _ in range(3):
                step(prm)
            torch.cuda.synchronize(dev)
            if world > 1:
                dist.barrier()
            ev0.record(stream)
            for _ in range(args.steps):
                step(prm)
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            v_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
            v_plan = clp.grpo_get_plan(N, D, V, T, prm)
            v_exec = (EXECUTED_NDV[f] + (2.0 if args.with_dw else 0.0)) * D * V * p.n_valid
            variants.append({
                "backward": FORM_NAMES[f], "ms_per_step": v_ms,
                "value": world * p.n_valid / (v_ms / 1e3),
                "tflops_executed": v_exec / (v_ms / 1e3) / 1e12,
                "workspace_bytes": v_plan["workspace_bytes"], "chunk_rows": v_plan["chunk_rows"],
                "vocab_block": v_plan["vocab_block"],
                "launches_per_call": v_plan["launches_loss"] + (
                    v_plan["n_chunks"] * v_plan["n_vocab_blocks"] if args.with_dw else 0)})

    # Forward alone (one logit GEMM launch + finalize), timed on the same stream.
    fwd_ms = None
    if rank == 0:
        for _ in range(3):
            clp.grpo_logp_fwd(p.hidden, p.weight, p.ids, params=params, workspace=ws, logp=logp)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        reps = max(5, args.steps // 2)
        for _ in range(reps):
            clp.grpo_logp_fwd(p.hidden, p.weight, p.ids, params=params, workspace=ws, logp=logp)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        fwd_ms = ev0.elapsed_time(ev1) / reps

    # End to end through the public API with host buffers: pinned H2D of the
    # step's inputs, the call, D2H of its results (loss, dH), every step.
    e2e = None
    if not args.no_e2e:
        # End to end through the public API with host buffers. Every step copies
        # its inputs from pinned host memory and reads its results (loss, dH)
        # back; a copy stream overlaps step i+1's inputs and step i-1's results
        # with step i's compute, on two sets of device buffers.
        host_in = [p.hidden.cpu().pin_memory(), p.ids.cpu().pin_memory(),
                   p.mask.cpu().pin_memory(), old.cpu().pin_memory(), ref.cpu().pin_memory(),
                   p.adv.cpu().pin_memory()]
        dev_in = [[torch.empty_like(x, device=dev) for x in host_in] for _ in range(2)]
        loss_d = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(2)]
        dH_d = [torch.empty(N, D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        loss_h = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
        dH_h = [torch.empty(N, D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        h2d_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        d2h_done = [torch.cuda.Event() for _ in range(2)]

        def run_e2e(n_steps):
            for i in range(n_steps):
                b = i & 1
                with torch.cuda.stream(h2d_s):
                    if i >= 2:
                        h2d_s.wait_event(comp_done[b])  # step i-2 is done with inputs b
                    for d_, h_ in zip(dev_in[b], host_in):
                        d_.copy_(h_, non_blocking=True)
                    h2d_done[b].record(h2d_s)
                stream.wait_event(h2d_done[b])
                if i >= 2:
                    stream.wait_event(d2h_done[b])  # step i-2's outputs are read out
                x = dev_in[b]
                clp.grpo_loss_fwd_bwd(x[0], p.weight, x[1], x[2], x[3], x[4], x[5], T,
                                      params=params, workspace=ws, loss=loss_d[b], logp=None,
                                      dH=dH_d[b], want_logp=False)
                comp_done[b].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(comp_done[b])
                    loss_h[b].copy_(loss_d[b], non_blocking=True)
                    dH_h[b].copy_(dH_d[b], non_blocking=True)
                    d2h_done[b].record(d2h_s)
            torch.cuda.synchronize(dev)

        run_e2e(3)
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        run_e2e(args.steps)
        e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.steps)
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        d2h = loss_h[0].numel() * 4 + dH_h[0].numel() * 2
        e2e = {"value": world * valid / (e_ms / 1e3), "unit": "tokens/s",
               "ms_per_step": e_ms, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "note": "pinned host hidden/ids/mask/old/ref/adv in and loss + dH out every "
                       "step, overlapped with compute on H2D and D2H copy streams "
                       "(double-buffered); "
                       "lm_head W resident on the device; host wall clock around the "
                       "synchronised steps"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    fl = flops_per_token(D, V) * valid
    tflops = fl / (ms_max / 1e3) / 1e12
    # Executed tensor work: 6NDV with the recomputed backward, 4NDV when the
    # backward reads the stored fp16 logits instead of a second logit GEMM.
    # With dW the single pass runs as the recomputed form (it never forms G).
    run_form = "recompute" if (form == "single_pass" and args.with_dw) else form
    fl_exec = (EXECUTED_NDV[run_form] + (2.0 if args.with_dw else 0.0)) * D * V * valid
    tflops_exec = fl_exec / (ms_max / 1e3) / 1e12
    peak_sus = peaks["bf16_tflops_sustained"]
    peak_burst = peaks["bf16_tflops"]
    rec = recorded_traffic(p.name, run_form)
    # The dominant kernel (most device time), timed live; its peak is the burst
    # one (a call lasts milliseconds). The call as a whole beside it.
    roofline = kernel_roofline(kernel_times, timed_calls, D, V, valid, peaks, rec,
                               ms_max if world == 1 else None) or {}
    roofline["peak_source"] = "%s (%s)" % (peak_src, "bf16 cuBLAS burst" if roofline.get(
        "bound") == "tensor" else "STREAM-style copy")
    roofline["timing"] = ("CUDA events recorded by the library around each launch on the "
                          "launch's own stream, over the %d timed calls" % timed_calls)
    roofline["traffic_unit"] = "DRAM bytes per launch (ncu dram__bytes_read.sum + write.sum)"
    roofline["call"] = {
        "scope": "grpo_loss_fwd_bwd: %d launches per call, %d chunks x %d vocab blocks" % (
            plan["launches_loss"], plan["n_chunks"], plan["n_vocab_blocks"]),
        "bound": "tensor", "achieved": tflops_exec, "peak": peak_burst, "unit": "TFLOP/s",
        "frac": tflops_exec / peak_burst, "frac_of_sustained_peak": tflops_exec / peak_sus,
        "counted_tflops_6NDV": tflops,
        "counted_note": "6NDV counted flops per second; the stored backward executes 4NDV, "
                        "so this rate is not a utilisation", "flops_per_call": fl_exec,
        "traffic": None if rec is None else rec.get("dram_bytes_per_call"),
        "traffic_unit": "DRAM bytes per call"}
    launches_per_call = sum(k["launches"] for k in kernel_times) / timed_calls
    out = {
        "metric": METRIC,
        "value": world * valid / (ms_max / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": p.name, "n_tokens": N, "valid_tokens": valid, "hidden": D,
            "vocab": V, "seq_len": T, "completions": p.n_seqs,
            "chunk_rows": plan["chunk_rows"], "vocab_block": plan["vocab_block"],
            "l2": "inputs larger than L2 (W %.2f GB, hidden %.0f MB); no flush" % (
                V * D * 2 / 1e9, N * D * 2 / 1e6),
            "parallelism": "replicas: one independent batch per GPU" if world > 1 else "1 GPU",
        },
        "tflops": tflops,
        "tflops_executed": tflops_exec,
        "pct_bf16_peak": 100.0 * tflops_exec / peak_burst,
        "pct_bf16_peak_note": "executed flops over the measured burst bf16 peak",
        "backward_choice": choice,
        "backward": FORM_NAMES[run_form] + (
            ", G formed inside the dH GEMM" if stored and plan["g_in_dh_gemm"]
            and not args.with_dw else ", G formed in its own pass" if stored else "") + (
            " + lm_head dW" if args.with_dw else ""),
        "variants": variants,
        "roofline": roofline,
        "fwd_only": None if fwd_ms is None else {
            "ms": fwd_ms, "tflops": 2.0 * D * V * N / (fwd_ms / 1e3) / 1e12,
            "frac_of_burst_peak": 2.0 * D * V * N / (fwd_ms / 1e3) / 1e12 / peak_burst,
            "scope": "grpo_logp_fwd: logit GEMM + finalize over all N rows"},
        "e2e": e2e,
        "clocks": clocks.summary(),
        "gpu_launches": launches_per_call * args.steps,
        "gpu_launches_source": "counted by the library's launch timing (%g per call)" % (
            launches_per_call),
        "workspace_bytes": plan["workspace_bytes"],
        "cpu_baseline": None,
    }
    if world == 1 and not args.no_cpu_baseline:
        step()  # the outputs of one headline call, for the parity check
        torch.cuda.synchronize(dev)
        def masked_loss(mask2):
            loss2 = torch.empty(1, dtype=torch.float32, device=dev)
            dH2 = torch.empty_like(dH)
            clp.grpo_loss_fwd_bwd(p.hidden, p.weight, p.ids, mask2.to(dev), old, ref, p.adv, T,
                                  params=params, workspace=ws, loss=loss2, logp=None, dH=dH2,
                                  want_logp=False)
            return float(loss2.item())

        n, t, parity = oracle_rows_per_second(p, args.cpu_seconds, args.seed, None,
                                              gpu=(old, ref, logp, dH), masked_loss=masked_loss)
        out["cpu_baseline"] = {
            "value": n / t, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} seeded valid rows of {p.name} (logp, g, dH per row; 6DV fp64 "
                      f"flops each), {t:.1f} s on the host cores (numpy/OpenBLAS threads)",
            "parity_vs_gpu": parity}
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# -------------------------------------------------------- budget sweep ----

def run_budget_sweep(args):
    """Workspace budget against call time: for each budget, the library's
    automatic choice and the three forced backward forms, each with the
    largest plan the budget allows. One JSON line per (budget, form); a form that does
    not fit a budget is reported as such."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as clp
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    p = synth.make_problem(args.workload, seed=args.seed, device=dev)
    torch.cuda.empty_cache()
    N, D, V, T = p.n_tokens, p.hidden_size, p.vocab, p.seq_len
    old = torch.full((N,), -math.log(V), device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    dH = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(3, args.steps)
    for gb in [float(x) for x in args.budget_sweep.split(",") if x.strip()]:
        limit = int(gb * (1 << 30))
        for form in ("auto", "stored", "single_pass", "recompute"):
            params = clp.make_params(p.eps_low, p.eps_high, p.beta,
                                     flags=FORM_FLAGS[form], workspace_limit_bytes=limit)
            row = {"workload": p.name, "budget_gb": gb, "form": form}
            try:
                nbytes = clp.grpo_workspace_size(N, D, V, T, params)
                plan = clp.grpo_get_plan(N, D, V, T, params)
            except clp.GrpoError as e:
                row["fits"] = False
                row["why"] = str(e)
                print(json.dumps(row), flush=True)
                continue
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

            def call():
                clp.grpo_loss_fwd_bwd(p.hidden, p.weight, p.ids, p.mask, old, old, p.adv, T,
                                      params=params, workspace=ws, loss=loss, logp=None, dH=dH,
                                      want_logp=False)
            for _ in range(max(args.warmup, 3)):
                call()
            torch.cuda.synchronize(dev)
            assert clp.grpo_read_device_status(ws) == 0
            ev0.record(stream)
            for _ in range(reps):
                call()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            ms = ev0.elapsed_time(ev1) / reps
            row.update({"fits": True, "workspace_bytes": nbytes,
                        "backward": form_of(plan),
                        "chunk_rows": plan["chunk_rows"], "n_chunks": plan["n_chunks"],
                        "vocab_block": plan["vocab_block"], "ms_per_call": ms,
                        "tokens_per_s": p.n_valid / (ms / 1e3)})
            print(json.dumps(row), flush=True)
            del ws
            torch.cuda.empty_cache()


# ----------------------------------------------------------- reference ----

def run_reference(args):
    # The oracle runs on rank 0's host cores only; other ranks exit without work.
    _, rank, _ = rank_env()
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    import synth

    p = synth.make_problem(args.workload, seed=args.seed, device="cpu")
    W64 = p.weight.float().numpy().astype(np.float64)
    valid = torch.nonzero(p.mask != 0).flatten().numpy()
    base = torch.full((p.n_tokens,), -math.log(p.vocab))
    old, ref = p.old_ref(base)
    M = float(len(valid))
    rng = np.random.default_rng(args.seed)
    # Rows per step: about 3 s of oracle work, calibrated on 16 rows after a
    # first call that pays the one-time costs (thread pool start-up, page-in).
    oracle.rows_fwd_bwd(p.hidden, W64, p.ids.numpy(), valid[:4], old, ref, p.adv, p.seq_len, M)
    t0 = time.perf_counter()
    oracle.rows_fwd_bwd(p.hidden, W64, p.ids.numpy(), valid[:16], old, ref, p.adv, p.seq_len, M)
    per_row = (time.perf_counter() - t0) / 16
    rows_per_step = int(max(4, min(len(valid), 3.0 / max(per_row, 1e-6))))

    def step():
        rows = np.sort(rng.choice(valid, size=rows_per_step, replace=False))
        oracle.rows_fwd_bwd(p.hidden, W64, p.ids.numpy(), rows, old, ref, p.adv, p.seq_len, M,
                            p.eps_low, p.eps_high, p.beta)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = rows_per_step / dt
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": p.name, "n_tokens": p.n_tokens, "hidden": p.hidden_size,
                   "vocab": p.vocab, "seq_len": p.seq_len},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle",
                         "sample": f"{rows_per_step} seeded valid rows per step of {p.name}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    a = parse_args()
    if a.record_traffic:
        # "auto" names the form a call takes without a budget: stored.
        r = record_traffic(a.record_traffic, a.workload,
                           "stored" if a.backward == "auto" else a.backward, a.record_command)
        print(json.dumps({k: r.get(k) for k in ("workload", "backward", "dram_bytes_per_call",
                                                "launches_per_call", "ncu_time_ms_per_call")}))
    elif a.impl == "reference":
        run_reference(a)
    elif a.budget_sweep:
        run_budget_sweep(a)
    else:
        run_ours(a)

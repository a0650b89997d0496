#!/usr/bin/env python
"""Decode-step benchmark of the OSCAR two-bit KV path on GB300.

Workload (Qwen3-8B-shaped single layer): batch 1, 32 query heads, 8 KV heads
(GQA 4), head_dim 128, context 100,000 tokens = 64 BF16 sink + 99,680 INT2
history (16-token pages, fp16 scale/zero per 128-channel group) + 256 BF16
recent.  Synthetic seeded data: N(0,1) with 4 outlier channels x20 per KV
head; rotations and clip thresholds built by the library from 4096 seeded
calibration queries and 2048 calibration keys/values per KV head.

One step = the whole hot path once: oscar_quantize_append_overlapped (the
oldest recent token of every KV head is rotated, clipped, quantised, packed
into history, and the new token written into the freed ring slot; its loads
and arithmetic overlap the previous layer copy's decode) + oscar_decode_attention
(q pre-rotation, INT2 split-KV scan, BF16 sink/recent scan, merge and output
rotation).  The step is replayed from a steady state (lengths do not advance,
so every step does identical work).  Steps cycle over several independent
copies of the layer cache whose total size exceeds 3x the L2 cache, so no
step reads its inputs from L2 (inputs larger than L2; no flush needed).

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference]
  python bench.py --workload qwen3-4b-36layer-b28-100k | qwen3-32b-layer-b64-ragged-prefix |
                  bulk-demote-128k-36layer

`--impl reference` times the float64 CPU oracle on this host instead.  The
other `--workload`s measure the larger stated workloads (one JSON line each):
a 36-layer decode step of 28 requests at 100k context, a batch-64 GQA-8
layer with ragged contexts and a shared 32k prefix, and the bulk demotion of
a 128k-token prefill followed by batch-1 decode over it.
"""
from __future__ import annotations

import argparse
import copy
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = dict(workload="qwen3-8b-layer-decode-100k", batch=1, n_q_heads=32, n_kv_heads=8,
                head_dim=128, ctx=100_000, sink=64, recent=256, page_tokens=16, group_k=128, group_v=128,
                codebook="uniform", seed=1002)
METRIC = "decode-attn tokens/s at 100k ctx (1 layer, Qwen3-8B shape)"
UNIT = "tokens/s"
EXTRA_WORKLOADS = {
    # 36-layer decode step: per layer one demotion per request + decode
    "qwen3-4b-36layer-b28-100k": dict(batch=28, n_q_heads=32, n_kv_heads=8, ctx=100_000, layers=36,
                                      seed=1003, distinct_layers=2),
    # one GQA-8 layer, contexts U[8k, 128k], first 32k tokens a shared prefix
    "qwen3-32b-layer-b64-ragged-prefix": dict(batch=64, n_q_heads=64, n_kv_heads=8, ctx_lo=8192,
                                              ctx_hi=131_072, shared=32_768, layers=1, seed=1004,
                                              distinct_layers=2),
    # rotate-clip-quantise-pack of a 128k-token prefill (8 KV heads, 36
    # layers), then batch-1 GQA-4 decode over the 128k history
    "bulk-demote-128k-36layer": dict(batch=1, n_q_heads=32, n_kv_heads=8, ctx=131_072, layers=36,
                                     seed=1005, distinct_layers=2),
}
# calibration covariance on the device: C = X^T X / N over 2^20 bf16 rows of
# 128 values (the C_Q / C_S accumulation of one KV head)
CALIB_WORKLOAD = "calib-covariance-1m"
VCALIB_WORKLOAD = "calib-value-covariance-8kv"
RING_START = 1     # ring slot of the oldest recent token in the steady state
CACHE_TENSORS = ("pages", "page_table", "hist_len", "sink_k", "sink_v", "sink_len", "recent_k",
                 "recent_v", "recent_len", "recent_start", "r_k", "r_v", "dev_status")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="oscar", choices=["oscar", "reference"])
    ap.add_argument("--cpu-baseline-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--reps", type=int, default=20, help=argparse.SUPPRESS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD["workload"],
                    choices=[WORKLOAD["workload"]] + sorted(EXTRA_WORKLOADS) + [CALIB_WORKLOAD, VCALIB_WORKLOAD])
    ap.add_argument("--rotation", default="oscar", choices=["oscar", "canalized32"],
                    help="R_K/R_V of the default workload: the OSCAR eigenbasis rotation, or the OScaR "
                         "block-diagonal one (Hadamard groups of 32 channels)")
    ap.add_argument("--quant-group", default="128,128",
                    choices=["%d,%d" % (a, b) for a in (32, 64, 128) for b in (32, 64, 128)],
                    help="quantisation group sizes of K and V (channels), for every GPU workload")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests of a --workload other than the default (0: the workload's own); a smaller "
                         "batch of the same kernel, for profiler captures")
    ap.add_argument("--codebook", default="uniform", choices=["uniform", "lloyd-max"],
                    help="code levels: the uniform scale/zero grid, or per-layer Lloyd-Max levels fitted on "
                         "the calibration rows (one quantisation group per vector)")
    args = ap.parse_args()
    WORKLOAD["group_k"], WORKLOAD["group_v"] = (int(x) for x in args.quant_group.split(","))
    WORKLOAD["codebook"] = args.codebook
    if args.codebook != "uniform" and (WORKLOAD["group_k"], WORKLOAD["group_v"]) != (128, 128):
        ap.error("--codebook lloyd-max takes one quantisation group per vector")
    if args.codebook != "uniform" and args.workload != WORKLOAD["workload"]:
        ap.error("--codebook lloyd-max applies to the default workload")
    return args


def _split(ctx):
    s = min(ctx, WORKLOAD["sink"])
    r = min(ctx - s, WORKLOAD["recent"])
    return s, ctx - s - r, r


def bytes_per_decode():
    """Algorithmic HBM bytes of one decode launch on the workload (per step)."""
    w = WORKLOAD
    _, hist, _ = _split(w["ctx"])
    d = w["head_dim"]
    per_hist_token = w["n_kv_heads"] * (2 * (d // 4) + 4 * (d // w["group_k"]) + 4 * (d // w["group_v"]))
    bf16 = (w["sink"] + w["recent"]) * w["n_kv_heads"] * 2 * w["head_dim"] * 2
    table = -(-hist // w["page_tokens"]) * 4
    io = w["n_q_heads"] * w["head_dim"] * (2 + 4)
    return hist * per_hist_token + bf16 + table + io


def _group_label():
    w = WORKLOAD
    return w["group_k"] if w["group_k"] == w["group_v"] else "k%d/v%d" % (w["group_k"], w["group_v"])


def _config_json(extra=None):
    w = WORKLOAD
    s, h, r = _split(w["ctx"])
    cfg = {"workload": w["workload"], "batch": w["batch"], "n_q_heads": w["n_q_heads"],
           "n_kv_heads": w["n_kv_heads"], "head_dim": w["head_dim"], "ctx": w["ctx"],
           "sink_bf16": s, "history_int2": h, "recent_bf16": r, "page_tokens": w["page_tokens"],
           "quant_group": _group_label(), "codebook": w["codebook"], "parallelism": "replicas"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------- oracle leg

def _oracle_sample_setup(head=0):
    """Inputs of one KV head (4 query heads) of the workload for the oracle."""
    import numpy as np
    import oracle as O
    import synth
    w = WORKLOAD
    seed = w["seed"]
    outl = synth.outlier_channels(seed, 0, w["n_kv_heads"])[head:head + 1]
    cal = synth.calibration_set(seed, 0, head, outl[0], n_q=4096, n_k=2048)
    rk = O.rotation_from_covariance(O.query_covariance(cal["q"]))
    rv = O.rotation_from_covariance(O.value_covariance(cal["q"], cal["k"], cal["v"]))
    tau_k = O.clip_threshold(cal["k"] @ rk)
    tau_v = O.clip_threshold(cal["v"] @ rv)
    s, h, r = _split(w["ctx"])
    k = synth.activations(seed, (0, head, 0), w["ctx"] + 1, outl).astype(np.float64)
    v = synth.activations(seed, (0, head, 1), w["ctx"] + 1, outl).astype(np.float64)
    g = w["n_q_heads"] // w["n_kv_heads"]
    q = synth.activations(seed, (0, head, 2), 1, np.repeat(outl, g, axis=0))[0].astype(np.float64)
    hist = {}
    if w["codebook"] != "uniform":
        # the oracle's own Lloyd-Max fit on this head's calibration rows
        hist["levels_k"] = O.fit_codebook(cal["k"], rk, tau_k)
        hist["levels_v"] = O.fit_codebook(cal["v"], rv, tau_v)
    for name, x, rot, tau in (("k", k, rk, tau_k), ("v", v, rv, tau_v)):
        c, sc, ze = _oracle_demote(O, x[s:s + h - 1, 0], rot, tau, w["group_" + name],
                                   hist.get("levels_" + name))
        hist["codes_" + name], hist["scale_" + name], hist["zero_" + name] = c[:, None], sc[:, None], ze[:, None]
    return dict(O=O, np=np, q=q, k=k, v=v, rk=rk, rv=rv, tau_k=tau_k, tau_v=tau_v, hist=hist, s=s, h=h, r=r)


def _oracle_demote(O, x, r, tau, group, levels=None):
    """The oracle's demotion of rows x with one or several quantisation groups,
    or with codebook levels."""
    if levels is not None:
        return O.quantize_codebook(O.rotate(x, r), tau, levels)
    if group == WORKLOAD["head_dim"]:
        return O.demote(x, r, tau)
    return O.quantize_groups(O.rotate(x, r), tau, group)


def _oracle_step(st, n_hist=None):
    """One decode step of one KV head, by the oracle: demote the oldest recent
    token into history, then attend over sink | history | recent.  `n_hist`
    limits the history to its first n_hist - 1 stored tokens plus the demoted
    one (a bounded sample; cost is linear in the history length)."""
    O, np = st["O"], st["np"]
    s, h = st["s"], st["h"]
    keep = (h - 1) if n_hist is None else max(0, min(h - 1, n_hist - 1))
    old = st["hist"]
    ck, sk, zk = _oracle_demote(O, st["k"][s + h - 1, 0][None], st["rk"], st["tau_k"], WORKLOAD["group_k"],
                                old.get("levels_k"))
    cv, sv, zv = _oracle_demote(O, st["v"][s + h - 1, 0][None], st["rv"], st["tau_v"], WORKLOAD["group_v"],
                                old.get("levels_v"))
    hist = {"codes_k": np.concatenate([old["codes_k"][:keep], ck[:, None]]),
            "scale_k": np.concatenate([old["scale_k"][:keep], sk[:, None]]),
            "zero_k": np.concatenate([old["zero_k"][:keep], zk[:, None]]),
            "codes_v": np.concatenate([old["codes_v"][:keep], cv[:, None]]),
            "scale_v": np.concatenate([old["scale_v"][:keep], sv[:, None]]),
            "zero_v": np.concatenate([old["zero_v"][:keep], zv[:, None]])}
    for name in ("levels_k", "levels_v"):
        if name in old:
            hist[name] = old[name]
    k, v = st["k"], st["v"]
    return O.decode_attention(st["q"], k[:s], v[:s], hist, k[s + h:s + h + st["r"]],
                              v[s + h:s + h + st["r"]], st["rk"][None], st["rv"][None])


SAMPLE_DESC = ("one of the 8 KV heads (its 4 query heads) of a full decode step at 100k context "
               "(demotion of 1 token + attention over 64 + 99,680 INT2 + 256 tokens); "
               "step time extrapolated x8 to all KV heads")


def cpu_baseline_worker(reps):
    st = _oracle_sample_setup()
    _oracle_step(st)
    t0 = time.perf_counter()
    for _ in range(reps):
        _oracle_step(st)
    dt = (time.perf_counter() - t0) / reps
    # one whole step, every KV head in full (no extrapolation)
    heads = [st] + [_oracle_sample_setup(h) for h in range(1, WORKLOAD["n_kv_heads"])]
    t1 = time.perf_counter()
    for sh in heads:
        _oracle_step(sh)
    full = time.perf_counter() - t1
    print(json.dumps({"sample_seconds": dt, "reps": reps, "full_step_seconds": full}))


def _host_cpu():
    """(model name, logical cores) of this host."""
    import platform
    name = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    name = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not name:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    name = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return name or platform.machine(), os.cpu_count()


def _single_thread_env():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    return env


def cpu_baseline(reps=20):
    """The oracle timed on one host core in a fresh process (started before any GPU work)."""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-worker",
                        "--reps", str(reps), "--quant-group",
                        "%d,%d" % (WORKLOAD["group_k"], WORKLOAD["group_v"]), "--codebook", WORKLOAD["codebook"]],
                       capture_output=True, text=True, env=_single_thread_env(),
                       timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr[-400:]}
    res = json.loads(r.stdout.strip().splitlines()[-1])
    model, n_cpu = _host_cpu()
    full = res["full_step_seconds"]
    return {"value": WORKLOAD["batch"] / full, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "one whole decode step at 100k context, all %d KV heads in full (demotion of 1 token and "
                      "attention over 64 + 99,680 INT2 + 256 tokens per head), timed once"
                      % WORKLOAD["n_kv_heads"],
            "step_seconds": full,
            "per_head_step_seconds": res["sample_seconds"],
            "per_head_note": SAMPLE_DESC + "; %d timed repetitions" % res["reps"],
            "host_cpu": model, "host_logical_cores": n_cpu}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    st = _oracle_sample_setup()
    h = st["h"]
    # size the per-step sample so that warm-up + timed steps take about 150 s
    t1 = time.perf_counter()
    _oracle_step(st)
    full = time.perf_counter() - t1
    n_hist = h
    budget = 150.0 / max(args.steps + args.warmup, 1)
    if full > budget:
        n_hist = max(h // 64, int(h * budget / full))
    frac = n_hist / h
    for _ in range(args.warmup):
        _oracle_step(st, n_hist)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(st, n_hist)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    step = dt * WORKLOAD["n_kv_heads"] / frac
    value = WORKLOAD["batch"] / step
    sample = SAMPLE_DESC if n_hist == h else (
        SAMPLE_DESC + "; history cut to the first %d of %d tokens per step and scaled by %.2f"
        % (n_hist, h, 1 / frac))
    model, n_cpu = _host_cpu()
    # ms_per_step: what each timed step measured (one KV head, the history
    # sample above); value: that time extrapolated to a whole step
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config_json(),
            "extrapolation": {"measured_ms_per_sample_step": dt * 1e3,
                              "factor": WORKLOAD["n_kv_heads"] / frac,
                              "whole_step_ms": step * 1e3,
                              "note": "each timed step runs one of the %d KV heads%s; value = batch / whole_step"
                                      % (WORKLOAD["n_kv_heads"], "" if n_hist == h else
                                         " over the first %d of %d history tokens" % (n_hist, h))},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "host_cpu": model, "host_logical_cores": n_cpu},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------------------- GPU leg

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons around the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        import tempfile
        self.index = index
        self.proc = None
        # the raw samples go to a temporary file (OSCAR_CLOCKS_CSV keeps them
        # at a chosen path); the JSON line carries their summary
        self.path = os.environ.get("OSCAR_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), "oscar_clocks_%d.csv" % os.getpid())

    def start(self):
        if os.path.dirname(self.path):
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


def _code_only(src):
    """C++ source with comments removed and whitespace runs collapsed (string
    and character literals kept), so that a comment edit leaves it unchanged."""
    import re
    tok = re.compile(r'"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'|//[^\n]*|/\*.*?\*/', re.S)
    out = tok.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", src)
    return " ".join(out.split())


def _profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu capture record
    (profiles/split_kernel_qwen3-8b-layer-decode-100k.json, beside its
    summary), if it was taken on the current kernel sources (else None)."""
    import hashlib
    if (WORKLOAD["group_k"], WORKLOAD["group_v"]) != (128, 128) or WORKLOAD["codebook"] != "uniform":
        return None    # the capture covers the one-group, uniform-level kernel
    prof = os.path.join(ROOT, "profiles", "split_kernel_qwen3-8b-layer-decode-100k.json")
    try:
        with open(prof) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for f in rec.get("source_files", []):
        with open(os.path.join(ROOT, "bit_rotated_kv_split_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    if not rec.get("source_files") or rec.get("source_sha256") != h.hexdigest():
        return None
    return int(rec["traffic_bytes_per_launch"])


def _roofline_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over the ranks of the default
    process group (gloo with CPU tensors, NCCL with CUDA tensors)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu().tolist()]


def rotations_from_library(B, kind="oscar"):
    """Per-head R_K, R_V and per-layer taus, built by the library's host routines
    (kind "canalized32": the OScaR block-diagonal rotation for K and V)."""
    import numpy as np
    import synth
    w = WORKLOAD
    seed, n_kv = w["seed"], w["n_kv_heads"]
    outl = synth.outlier_channels(seed, 0, n_kv)
    rk, rv, ck, cv = [], [], [], []
    for hh in range(n_kv):
        cal = synth.calibration_set(seed, 0, hh, outl[hh], n_q=4096, n_k=2048)
        if kind == "canalized32":
            rk.append(B.oscar_build_canalized_rotation(w["head_dim"], 32))
            rv.append(B.oscar_build_canalized_rotation(w["head_dim"], 32))
        else:
            rk.append(B.oscar_build_rotation(cal["q"])[0])
            rv.append(B.oscar_build_rotation(B.oscar_score_weighted_rows(cal["q"], cal["k"], cal["v"]))[0])
        ck.append(cal["k"])
        cv.append(cal["v"])
    rk32 = np.stack(rk).astype(np.float32)
    rv32 = np.stack(rv).astype(np.float32)
    tau_k = B.oscar_clip_threshold(np.stack(ck), rk32.astype(np.float64))
    tau_v = B.oscar_clip_threshold(np.stack(cv), rv32.astype(np.float64))
    if w["codebook"] != "uniform":
        # Lloyd-Max levels of the layer from its heads' rotated calibration rows
        eye = np.eye(w["head_dim"])
        xk = np.concatenate([ck[i] @ rk32[i].astype(np.float64) for i in range(n_kv)])
        xv = np.concatenate([cv[i] @ rv32[i].astype(np.float64) for i in range(n_kv)])
        w["levels_k"] = [float(x) for x in B.oscar_fit_codebook(xk, eye, tau_k)]
        w["levels_v"] = [float(x) for x in B.oscar_fit_codebook(xv, eye, tau_v)]
    return rk32, rv32, tau_k, tau_v, outl


def build_layer(torch, B, dev, rot):
    """One layer cache of the workload on `dev`, history filled by the library's own demotion."""
    import synth
    from bit_rotated_kv_split_gb300.cache import LayerCache
    w = WORKLOAD
    seed, n_kv, bsz = w["seed"], w["n_kv_heads"], w["batch"]
    s, h, r = _split(w["ctx"])
    rk, rv, tau_k, tau_v, outl = rot
    table, n_pages = synth.page_table(seed, [h] * bsz, n_extra_pages=1)
    cache = LayerCache(bsz, w["n_q_heads"], n_kv, table.shape[1], n_pages, torch.from_numpy(rk),
                       torch.from_numpy(rv), tau_k, tau_v, device=dev, quant_group_k=w["group_k"],
                       quant_group_v=w["group_v"], levels_k=w.get("levels_k"), levels_v=w.get("levels_v"))
    cache.page_table.copy_(torch.from_numpy(table))
    cache.max_hist = h
    chunk = 32768
    for b in range(bsz):
        for t0 in range(0, h, chunk):
            n = min(chunk, h - t0)
            xk = synth.activations_device(seed, (0, b, 0, t0), n, outl, dev)
            xv = synth.activations_device(seed, (0, b, 1, t0), n, outl, dev)
            pos = torch.arange(t0, t0 + n, dtype=torch.int32, device=dev)
            req = torch.full((n,), b, dtype=torch.int32, device=dev)
            B.oscar_quantize_append(cache.desc(h), xk.view(torch.uint16), xv.view(torch.uint16), n,
                                    n_kv * 128, None, req, pos, n)
    sk = synth.activations_device(seed, (1, 0), bsz * w["sink"], outl, dev)
    sv = synth.activations_device(seed, (1, 1), bsz * w["sink"], outl, dev)
    rk_ = synth.activations_device(seed, (1, 2), bsz * w["recent"], outl, dev)
    rv_ = synth.activations_device(seed, (1, 3), bsz * w["recent"], outl, dev)
    cache.sink_k.copy_(sk.view(cache.sink_k.shape))
    cache.sink_v.copy_(sv.view(cache.sink_v.shape))
    cache.recent_k.copy_(rk_.view(cache.recent_k.shape))
    cache.recent_v.copy_(rv_.view(cache.recent_v.shape))
    cache.hist_len.fill_(h)
    cache.sink_len.fill_(s)
    cache.recent_len.fill_(r)
    # the oldest recent token sits in ring slot 1; every step demotes it and
    # writes the new token into that slot.  Lengths and the ring start are
    # not advanced, so each step does identical work (attention does not
    # depend on where in the ring a token sits).
    cache.recent_start.fill_(RING_START)
    torch.cuda.synchronize()
    assert int(cache.dev_status.item()) == 0
    return cache


def clone_layer(layer):
    c = copy.copy(layer)
    for name in CACHE_TENSORS:
        setattr(c, name, getattr(layer, name).clone())
    return c


def run_gpu(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.reps)          # before any GPU work in this process
    import torch
    import torch.distributed as dist
    from bit_rotated_kv_split_gb300 import binding as B
    import synth
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOAD
    bsz, n_kv = w["batch"], w["n_kv_heads"]
    s, h, r = _split(w["ctx"])

    rot = rotations_from_library(B, args.rotation)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    layer0 = build_layer(torch, B, dev, rot)
    per_layer = layer0.pages.numel() + 4 * (layer0.sink_k.numel() + layer0.recent_k.numel())
    n_copies = max(2, math.ceil(3 * l2 / per_layer))
    layers = [layer0] + [clone_layer(layer0) for _ in range(n_copies - 1)]
    torch.cuda.synchronize()

    qo = synth.outlier_channels(w["seed"], 0, n_kv).repeat(w["n_q_heads"] // n_kv, axis=0)
    q = synth.activations_device(w["seed"], (2, 0), bsz, qo, dev).view(bsz, w["n_q_heads"], 128)
    new_k = synth.activations_device(w["seed"], (2, 1), bsz, rot[4], dev)
    new_v = synth.activations_device(w["seed"], (2, 2), bsz, rot[4], dev)
    out = torch.empty((bsz, w["n_q_heads"], 128), dtype=torch.float32, device=dev)
    # ring row of each request's oldest recent token (the one a step demotes)
    src = torch.tensor([b * w["recent"] + RING_START for b in range(bsz)], dtype=torch.int32, device=dev)
    dst_req = torch.arange(bsz, dtype=torch.int32, device=dev)
    dst_pos = torch.full((bsz,), h - 1, dtype=torch.int32, device=dev)
    descs = [L.desc(h) for L in layers]
    ws_bytes = B.oscar_decode_workspace_bytes(descs[0])
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)

    def demote(i, overlapped=True):
        # in a step the demotion follows the previous layer copy's decode,
        # which writes nothing it reads: its loads and arithmetic overlap that
        # kernel (the per-kernel timing below uses the plain entry point)
        L = layers[i]
        fn = B.oscar_quantize_append_overlapped if overlapped else B.oscar_quantize_append
        fn(descs[i], L.recent_k.view(torch.uint16), L.recent_v.view(torch.uint16),
           bsz * w["recent"], n_kv * 128, src, dst_req, dst_pos, bsz,
           new_k.view(torch.uint16), new_v.view(torch.uint16))

    def decode(i):
        B.oscar_decode_attention(descs[i], q, out, ws, ws_bytes)

    # CUDA graphs: one per layer copy holding a whole step (demotion +
    # decode), and two "kernel" graphs holding every copy's decode (resp.
    # demotion) back to back, for the per-kernel durations
    stream = torch.cuda.Stream()
    use_graphs = True
    g_step, g_chain, g_decode, g_demote = [], None, None, None
    try:
        with torch.cuda.stream(stream):
            for i in range(n_copies):
                demote(i)
                decode(i)
            torch.cuda.synchronize()
            for i in range(n_copies):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    demote(i)
                    decode(i)
                g_step.append(g)
            # every copy's step in order, as a serving loop replays all layers
            # (kernel to kernel edges are programmatic launches)
            g_chain = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_chain, stream=stream):
                for i in range(n_copies):
                    demote(i)
                    decode(i)
            g_decode, g_demote = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_decode, stream=stream):
                for i in range(n_copies):
                    decode(i)
            with torch.cuda.graph(g_demote, stream=stream):
                for i in range(n_copies):
                    demote(i, overlapped=False)
    except Exception as exc:  # graph capture unavailable: launch directly
        use_graphs = False
        sys.stderr.write("graph capture failed (%s); timing direct launches\n" % exc)
    torch.cuda.synchronize()

    def run_step(i):
        if use_graphs:
            g_step[i].replay()
        else:
            demote(i)
            decode(i)

    def run_steps(n):
        """n steps over the layer copies 0, 1, ... in order (whole chains, then single steps)."""
        if use_graphs:
            for _ in range(n // n_copies):
                g_chain.replay()
            for k in range(n % n_copies):
                g_step[k].replay()
        else:
            for k in range(n):
                run_step(k % n_copies)

    def run_all(graph, fn):
        if use_graphs:
            graph.replay()
        else:
            for i in range(n_copies):
                fn(i)

    K, W = args.steps, args.warmup
    clocks = Clocks(local)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    with torch.cuda.stream(stream):
        run_steps(W)
        torch.cuda.synchronize()
        clocks.start()
        t_pre = time.perf_counter()
        pre = 0
        while time.perf_counter() - t_pre < 1.0:      # same load before the timed region, for clock samples
            run_steps(7 * n_copies)
            pre += 7 * n_copies
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ev[0].record(stream)
        run_steps(K)
        ev[1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        # per-kernel durations: every copy's decode (then demotion) back to
        # back, repeated so that as many launches run as in the timed steps
        reps = max(1, K // n_copies)
        ev[2].record(stream)
        for _ in range(reps):
            run_all(g_decode, decode)
        ev[3].record(stream)
        for _ in range(reps):
            run_all(g_demote, lambda i: demote(i, overlapped=False))
        ev[4].record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
    total_ms = ev[0].elapsed_time(ev[1])
    decode_ms = ev[2].elapsed_time(ev[3]) / (reps * n_copies)
    demote_ms = ev[3].elapsed_time(ev[4]) / (reps * n_copies)
    t_step = total_ms / K / 1e3
    status = max(int(L.dev_status.item()) for L in layers)

    # end to end through the public API with pinned host buffers: one
    # oscar_decode_step per step brings its inputs (q, new K, new V: one
    # pinned staging buffer) to the device, demotes, decodes and writes the
    # output back to pinned host memory
    nq, nk = q.numel(), new_k.numel()
    inp = torch.empty(nq + 2 * nk, dtype=torch.bfloat16, device=dev)
    q_e, nk_e, nv_e = inp[:nq].view_as(q), inp[nq:nq + nk].view_as(new_k), inp[nq + nk:].view_as(new_v)
    inp_host = torch.cat([q.flatten(), new_k.flatten(), new_v.flatten()]).cpu().pin_memory()
    out_host = torch.empty(out.shape, dtype=torch.float32).pin_memory()

    sh = stream.cuda_stream     # the stream handle, passed to the calls

    in_bytes = inp.numel() * inp.element_size()
    rk16 = [L.recent_k.view(torch.uint16) for L in layers]
    rv16 = [L.recent_v.view(torch.uint16) for L in layers]
    nk16, nv16 = nk_e.view(torch.uint16), nv_e.view(torch.uint16)

    def step_e2e(i):
        # one library call: H2D copy of the step's inputs, demotion, decode,
        # D2H copy of the output; the demotion overlaps the previous call's
        # decode (another layer copy, whose writes go to out / out_host only)
        B.oscar_decode_step(descs[i], inp_host, inp, in_bytes, rk16[i], rv16[i], bsz * w["recent"], n_kv * 128,
                            src, dst_req, dst_pos, bsz, nk16, nv16, q_e, out, ws, ws_bytes, out_host, stream=sh,
                            flags=B.OSCAR_STEP_OVERLAP_PREVIOUS)

    ke = min(K, 500)
    with torch.cuda.stream(stream):
        for k in range(5):
            step_e2e(k % n_copies)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(ke):
            step_e2e(k % n_copies)
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3 / ke
    if world > 1:
        # the slowest rank sets the whole job's time
        t_step, e2e_s = max_over_ranks([t_step, e2e_s], dev)

    if rank == 0:
        peak, peak_kind = _roofline_peak()
        nbytes = bytes_per_decode()
        achieved = nbytes / (decode_ms / 1e3) / 1e9
        line = {
            "metric": METRIC, "value": world * bsz / t_step, "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": t_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int2/bf16 in, f32 accumulate",
            "data": "synthetic",
            "config": _config_json({"l2_policy": "inputs larger than L2: %d rotating layer caches of %.1f MB "
                                                 "(%.0f MB > 3x L2 %.0f MB)" % (n_copies, per_layer / 1e6,
                                                                                n_copies * per_layer / 1e6, l2 / 1e6),
                                    "cuda_graphs": use_graphs, "rotation": args.rotation}),
            "decode_ms": decode_ms, "demote_ms": demote_ms,
            "hbm_gbs_decode": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": _profiled_traffic(),
                         "kernel": "split_kernel (oscar_decode_attention, one launch per step)",
                         "algorithmic_bytes": nbytes, "peak_kind": peak_kind + " hbm_gbs"},
            "cpu_baseline": cpu,
            "e2e": {"value": world * bsz / e2e_s, "unit": UNIT,
                    "h2d_bytes_per_step": q.numel() * 2 + new_k.numel() * 2 + new_v.numel() * 2,
                    "d2h_bytes_per_step": out.numel() * 4},
            "gpu_launches": 2 * K,
            "kernel_timing": "decode_ms / demote_ms: %d back-to-back launches over the %d layer copies, "
                             "CUDA events on the launching stream" % (reps * n_copies, n_copies),
            "clocks": clk,
            "device_status": status,
            "host_wall_s": wall,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- larger stated workloads

def _rotations_for(B, seed, n_kv, layer):
    """R_K, R_V, tau_K, tau_V of one layer, built by the library from seeded calibration data."""
    import numpy as np
    import synth
    outl = synth.outlier_channels(seed, layer, n_kv)
    rk, rv, ck, cv = [], [], [], []
    for hh in range(n_kv):
        cal = synth.calibration_set(seed, layer, hh, outl[hh], n_q=4096, n_k=2048)
        rk.append(B.oscar_build_rotation(cal["q"])[0])
        rv.append(B.oscar_build_rotation(B.oscar_score_weighted_rows(cal["q"], cal["k"], cal["v"]))[0])
        ck.append(cal["k"])
        cv.append(cal["v"])
    rk32 = np.stack(rk).astype(np.float32)
    rv32 = np.stack(rv).astype(np.float32)
    tau_k = B.oscar_clip_threshold(np.stack(ck), rk32.astype(np.float64))
    tau_v = B.oscar_clip_threshold(np.stack(cv), rv32.astype(np.float64))
    return rk32, rv32, tau_k, tau_v, outl


def _build_batch_cache(torch, B, dev, rot, seed, layer, ctxs, n_q, n_kv, shared_hist=0):
    """Layer cache for requests of contexts `ctxs`; history demoted by the library.

    With `shared_hist`, the full history pages below it are one physical set
    shared by every request (demoted once)."""
    import synth
    from bit_rotated_kv_split_gb300.cache import LayerCache
    rk, rv, tau_k, tau_v, outl = rot
    splits = [_split(c) for c in ctxs]
    hist = [h for _, h, _ in splits]
    table, n_pages = synth.page_table(seed + 100 * layer, hist, n_extra_pages=1, shared_prefix_tokens=shared_hist)
    bsz = len(ctxs)
    cache = LayerCache(bsz, n_q, n_kv, table.shape[1], n_pages, torch.from_numpy(rk), torch.from_numpy(rv),
                       tau_k, tau_v, device=dev, quant_group_k=WORKLOAD["group_k"],
                       quant_group_v=WORKLOAD["group_v"])
    cache.page_table.copy_(torch.from_numpy(table))
    cache.max_hist = max(hist)
    n_shared_pages = 0
    if shared_hist:
        n_shared_pages = min(shared_hist // 16, max(h // 16 for h in hist))
    shared_tok = [min(n_shared_pages, h // 16) * 16 for h in hist]
    chunk = 32768
    done_shared = 0
    for b in range(bsz):
        lo = shared_tok[b] if done_shared >= shared_tok[b] else done_shared
        for t0 in range(lo, hist[b], chunk):
            n = min(chunk, hist[b] - t0)
            stream_b = 0 if t0 < shared_tok[b] else b
            xk = synth.activations_device(seed, (layer, stream_b, 0, t0), n, outl, dev)
            xv = synth.activations_device(seed, (layer, stream_b, 1, t0), n, outl, dev)
            pos = torch.arange(t0, t0 + n, dtype=torch.int32, device=dev)
            req = torch.full((n,), b, dtype=torch.int32, device=dev)
            B.oscar_quantize_append(cache.desc(max(hist) + 16), xk.view(torch.uint16), xv.view(torch.uint16), n,
                                    n_kv * 128, None, req, pos, n)
        done_shared = max(done_shared, shared_tok[b])
    cap_s, cap_r = WORKLOAD["sink"], WORKLOAD["recent"]
    sk = synth.activations_device(seed, (layer, 1, 0), bsz * cap_s, outl, dev)
    sv = synth.activations_device(seed, (layer, 1, 1), bsz * cap_s, outl, dev)
    rk_ = synth.activations_device(seed, (layer, 1, 2), bsz * cap_r, outl, dev)
    rv_ = synth.activations_device(seed, (layer, 1, 3), bsz * cap_r, outl, dev)
    cache.sink_k.copy_(sk.view(cache.sink_k.shape))
    cache.sink_v.copy_(sv.view(cache.sink_v.shape))
    cache.recent_k.copy_(rk_.view(cache.recent_k.shape))
    cache.recent_v.copy_(rv_.view(cache.recent_v.shape))
    cache.hist_len.copy_(torch.tensor(hist, dtype=torch.int32))
    cache.sink_len.copy_(torch.tensor([x for x, _, _ in splits], dtype=torch.int32))
    cache.recent_len.copy_(torch.tensor([x for _, _, x in splits], dtype=torch.int32))
    cache.recent_start.fill_(RING_START)
    torch.cuda.synchronize()
    assert int(cache.dev_status.item()) == 0
    unique_hist = n_shared_pages * 16 + sum(h - st for h, st in zip(hist, shared_tok))
    return cache, hist, unique_hist


def _hist_bytes_per_token(n_kv):
    """INT2 history bytes of one token (K and V codes, one (scale, zero) per group)."""
    return n_kv * (2 * (128 // 4) + 4 * (128 // WORKLOAD["group_k"]) + 4 * (128 // WORKLOAD["group_v"]))


def _decode_bytes(hist_tokens, ctx_tokens_bf16, n_q, n_kv, n_hist_pages):
    per_hist_token = _hist_bytes_per_token(n_kv)
    return (hist_tokens * per_hist_token + ctx_tokens_bf16 * n_kv * 2 * 128 * 2 + n_hist_pages * 4
            + n_q * 128 * 6)


def run_extra(args):
    import numpy as np
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    import synth
    cfg = EXTRA_WORKLOADS[args.workload]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n_q, n_kv, seed, L, nd = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["seed"], cfg["layers"], cfg["distinct_layers"]
    bsz = args.batch or cfg["batch"]
    K, W = args.steps, args.warmup
    peak, peak_kind = _roofline_peak()
    rots = [_rotations_for(B, seed, n_kv, i) for i in range(nd)]
    stream = torch.cuda.Stream()
    clocks = Clocks(0)
    line = {"n_gpus": 1, "steps": K, "warmup": W, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int2/bf16 in, f32 accumulate", "data": "synthetic"}

    if args.workload == "bulk-demote-128k-36layer":
        ctx = cfg["ctx"]
        s0, h, r0 = _split(ctx)
        caches, srcs = [], []
        for i in range(nd):
            c, _, _ = _build_batch_cache(torch, B, dev, rots[i], seed, i, [ctx], n_q, n_kv)
            caches.append(c)
            srcs.append((synth.activations_device(seed, (50 + i, 0), ctx, rots[i][4], dev),
                         synth.activations_device(seed, (50 + i, 1), ctx, rots[i][4], dev)))
        req = torch.zeros(h, dtype=torch.int32, device=dev)
        pos = torch.arange(h, dtype=torch.int32, device=dev)
        descs = [c.desc(h) for c in caches]
        q = synth.activations_device(seed, (60, 0), 1, rots[0][4].repeat(n_q // n_kv, axis=0), dev).view(1, n_q, 128)
        out = torch.empty((1, n_q, 128), dtype=torch.float32, device=dev)
        ws_bytes = B.oscar_decode_workspace_bytes(descs[0])
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)

        def demote_layer(i):
            # the prefill buffers from their first history token (row s0):
            # contiguous rows, no index
            xk, xv = srcs[i % nd]
            B.oscar_quantize_append(descs[i % nd], xk[s0:].view(torch.uint16), xv[s0:].view(torch.uint16),
                                    ctx - s0, n_kv * 128, None, req, pos, h)

        def decode(i):
            B.oscar_decode_attention(descs[i % nd], q, out, ws, ws_bytes)

        with torch.cuda.stream(stream):
            gd, gq = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            for i in range(2):
                demote_layer(i)
                decode(i)
            torch.cuda.synchronize()
            with torch.cuda.graph(gd, stream=stream):
                for i in range(L):
                    demote_layer(i)
            with torch.cuda.graph(gq, stream=stream):
                for i in range(2 * nd):
                    decode(i)
            for _ in range(W):
                gd.replay()
                gq.replay()
            torch.cuda.synchronize()
            clocks.start()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            for _ in range(K):
                gd.replay()
            e[1].record(stream)
            for _ in range(K):
                gq.replay()
            e[2].record(stream)
            torch.cuda.synchronize()
            clk = clocks.stop()
        t_bulk = e[0].elapsed_time(e[1]) / 1e3 / K            # 36 layers
        t_dec = e[1].elapsed_time(e[2]) / 1e3 / (K * 2 * nd)
        bulk_bytes = L * h * (n_kv * 2 * 128 * 2 + _hist_bytes_per_token(n_kv))
        dec_bytes = _decode_bytes(h, s0 + r0, n_q, n_kv, -(-h // 16))
        status = max(int(c.dev_status.item()) for c in caches)
        line.update({
            "metric": "bulk demotion GB/s (read + written) of a 128k-token prefill, 8 KV heads x 36 layers",
            "value": bulk_bytes / t_bulk / 1e9, "unit": "GB/s", "ms_per_step": t_bulk * 1e3,
            "config": {"workload": args.workload, "tokens": h, "n_kv_heads": n_kv, "head_dim": 128, "layers": L,
                       "quant_group": _group_label(),
                       "distinct_layers": nd, "l2_policy": "inputs larger than L2 (prefill buffers of %.0f MB per layer)"
                       % (ctx * n_kv * 128 * 2 * 2 / 1e6)},
            "roofline": {"bound": "hbm", "achieved": bulk_bytes / t_bulk / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": bulk_bytes / t_bulk / 1e9 / peak, "kernel": "demote_kernel (oscar_quantize_append)",
                         "algorithmic_bytes": bulk_bytes, "peak_kind": peak_kind + " hbm_gbs"},
            "decode_after": {"ms": t_dec * 1e3, "tokens_per_s": 1 / t_dec, "hbm_gbs": dec_bytes / t_dec / 1e9,
                             "frac": dec_bytes / t_dec / 1e9 / peak, "algorithmic_bytes": dec_bytes,
                             "context": ctx, "n_q_heads": n_q},
            "gpu_launches": K * (L + 2 * nd), "clocks": clk, "device_status": status})
        print(json.dumps(line))
        return

    # decode-step workloads
    if "ctx" in cfg:
        ctxs = [cfg["ctx"]] * bsz
    else:
        ctxs = [int(c) for c in synth.ragged_lengths(seed, bsz, cfg["ctx_lo"], cfg["ctx_hi"])]
    shared_hist = cfg.get("shared", 0)
    shared_hist = shared_hist - WORKLOAD["sink"] if shared_hist else 0
    caches, uniq = [], 0
    for i in range(nd):
        c, hist, uniq = _build_batch_cache(torch, B, dev, rots[i], seed, i, ctxs, n_q, n_kv, shared_hist)
        caches.append(c)
    g = n_q // n_kv
    q = synth.activations_device(seed, (70, 0), bsz, rots[0][4].repeat(g, axis=0), dev).view(bsz, n_q, 128)
    new_k = synth.activations_device(seed, (70, 1), bsz, rots[0][4], dev)
    new_v = synth.activations_device(seed, (70, 2), bsz, rots[0][4], dev)
    out = torch.empty((bsz, n_q, 128), dtype=torch.float32, device=dev)
    src = torch.tensor([b * WORKLOAD["recent"] + RING_START for b in range(bsz)], dtype=torch.int32, device=dev)
    dst_req = torch.arange(bsz, dtype=torch.int32, device=dev)
    dst_pos = torch.tensor(hist, dtype=torch.int32, device=dev)        # private tail slot of each request
    descs = [c.desc(max(hist) + 16) for c in caches]
    ddescs = [c.desc(max(hist)) for c in caches]
    ws_bytes = B.oscar_decode_workspace_bytes(ddescs[0])
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)

    def demote(i):
        # follows the previous layer's decode, which writes only out and ws
        c = caches[i % nd]
        B.oscar_quantize_append_overlapped(descs[i % nd], c.recent_k.view(torch.uint16),
                                           c.recent_v.view(torch.uint16), bsz * WORKLOAD["recent"], n_kv * 128,
                                           src, dst_req, dst_pos, bsz, new_k.view(torch.uint16),
                                           new_v.view(torch.uint16))

    def decode(i):
        B.oscar_decode_attention(ddescs[i % nd], q, out, ws, ws_bytes)

    with torch.cuda.stream(stream):
        for i in range(nd):
            demote(i)
            decode(i)
        torch.cuda.synchronize()
        g_step, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=stream):
            for i in range(L):
                demote(i)
                decode(i)
        with torch.cuda.graph(g_dec, stream=stream):
            for i in range(max(L, 2 * nd)):
                decode(i)
        for _ in range(W):
            g_step.replay()
        torch.cuda.synchronize()
        clocks.start()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        for _ in range(K):
            g_step.replay()
        e[1].record(stream)
        for _ in range(K):
            g_dec.replay()
        e[2].record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
    t_step = e[0].elapsed_time(e[1]) / 1e3 / K
    t_dec = e[1].elapsed_time(e[2]) / 1e3 / (K * max(L, 2 * nd))
    bf16_tok = sum(sum(_split(c)[0::2]) for c in ctxs)
    logical = _decode_bytes(sum(hist), bf16_tok, n_q * bsz, n_kv, sum(-(-h // 16) for h in hist))
    unique = _decode_bytes(uniq, bf16_tok, n_q * bsz, n_kv, sum(-(-h // 16) for h in hist))
    status = max(int(c.dev_status.item()) for c in caches)
    metric = ("36-layer decode-step tokens/s (Qwen3-4B shape, batch %d, 100k ctx, 1 demotion per request-layer)"
              if L > 1 else "decode tokens/s (Qwen3-32B layer, batch %d, ragged 8k-128k ctx, shared 32k prefix)") % bsz
    line.update({
        "metric": metric, "value": bsz / t_step, "unit": "tokens/s", "ms_per_step": t_step * 1e3,
        "config": {"workload": args.workload, "batch": bsz, "n_q_heads": n_q, "n_kv_heads": n_kv, "head_dim": 128,
                   "layers": L, "distinct_layers": nd, "ctx_min": min(ctxs), "ctx_max": max(ctxs),
                   "quant_group": _group_label(),
                   "ctx_mean": sum(ctxs) / bsz, "shared_prefix_tokens": cfg.get("shared", 0),
                   "l2_policy": "inputs %s than L2: %d distinct layer caches, each read %.0f MB per decode "
                                "(unique) against 129 MB of L2" % ("larger" if unique > 129e6 else "NOT larger",
                                                                    nd, unique / 1e6), "cuda_graphs": True},
        "decode_ms": t_dec * 1e3,
        "roofline": {"bound": "hbm", "achieved": unique / t_dec / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": unique / t_dec / 1e9 / peak, "kernel": "split_kernel (oscar_decode_attention)",
                     "algorithmic_bytes": unique, "logical_bytes": logical, "peak_kind": peak_kind + " hbm_gbs"},
        "logical_gbs": logical / t_dec / 1e9,
        "gpu_launches": K * 2 * L, "clocks": clk, "device_status": status})
    print(json.dumps(line))


def run_calibration(args):
    """oscar_covariance over 2^20 seeded bf16 rows (256 MB, larger than L2): one
    covariance per step, timed with CUDA events on the launching stream."""
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = 1 << 20
    outl = synth.outlier_channels(1006, 0, 1)
    x = synth.activations_device(1006, (70, 0), n, outl, dev).view(n, 128).contiguous()
    c = torch.empty((128, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(B.oscar_covariance_workspace_bytes(n), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    K, W = args.steps, args.warmup
    clocks = Clocks(0)
    with torch.cuda.stream(stream):
        for _ in range(max(W, 3)):
            B.oscar_covariance(x, c, ws)
        torch.cuda.synchronize()
        clocks.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            B.oscar_covariance(x, c, ws)
        e1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
    t = e0.elapsed_time(e1) / K / 1e3
    peak, peak_kind = _roofline_peak()
    nbytes = n * 128 * 2
    flops = 2.0 * n * 128 * 128
    gbs = nbytes / t / 1e9
    print(json.dumps({
        "metric": "calibration covariance GB/s (2^20 bf16 rows of 128, C = X^T X / N)", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 accumulate", "data": "synthetic",
        "config": {"workload": CALIB_WORKLOAD, "rows": n, "d": 128, "l2_policy": "input 256 MB > L2"},
        "tflops": flops / t / 1e12,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "kernel": "covariance_partial_kernel (oscar_covariance)", "algorithmic_bytes": nbytes,
                     "peak_kind": peak_kind + " hbm_gbs"},
        "gpu_launches": 2 * K, "clocks": clk}))


def run_value_calibration(args):
    """oscar_value_covariance for the 8 KV heads of one layer (4096 seeded
    calibration queries and 2048 keys/values per head, the calibration sets
    the default workload's rotations come from): one layer per step, the
    heads on streams of their own that fork from and join the timed stream,
    timed with CUDA events on that stream.  The roofline is the tensor pipe's
    (the work is two dense contractions per head)."""
    import numpy as np
    import torch
    from bit_rotated_kv_split_gb300 import binding as B
    import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    seed, n_kv, n_q, n_k = WORKLOAD["seed"], WORKLOAD["n_kv_heads"], 4096, 2048
    outl = synth.outlier_channels(seed, 0, n_kv)
    qs, ks, vs = [], [], []
    for hh in range(n_kv):
        cal = synth.calibration_set(seed, 0, hh, outl[hh], n_q=n_q, n_k=n_k)
        qs.append(torch.from_numpy(np.ascontiguousarray(cal["q"])).to(torch.bfloat16).to(dev))
        ks.append(torch.from_numpy(np.ascontiguousarray(cal["k"])).to(torch.bfloat16).to(dev))
        vs.append(torch.from_numpy(np.ascontiguousarray(cal["v"])).to(torch.bfloat16).to(dev))
    c = torch.empty((n_kv, 128, 128), dtype=torch.float32, device=dev)
    # the heads are independent: one stream and one workspace per head, so
    # their kernels run side by side (a head alone fills a fraction of the SMs)
    wss = [torch.empty(B.oscar_value_covariance_workspace_bytes(n_q), dtype=torch.uint8, device=dev)
           for _ in range(n_kv)]
    stream = torch.cuda.Stream()
    head_streams = [torch.cuda.Stream() for _ in range(n_kv)]
    K, W = args.steps, args.warmup

    def layer():
        ev = torch.cuda.Event()
        ev.record(stream)
        for hh in range(n_kv):
            hs = head_streams[hh]
            hs.wait_event(ev)
            B.oscar_value_covariance(qs[hh], ks[hh], vs[hh], c[hh], wss[hh], stream=hs.cuda_stream)
        for hs in head_streams:
            done = torch.cuda.Event()
            done.record(hs)
            stream.wait_event(done)

    clocks = Clocks(0)
    with torch.cuda.stream(stream):
        for _ in range(max(W, 3)):
            layer()
        torch.cuda.synchronize()
        clocks.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            layer()
        e1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
    t = e0.elapsed_time(e1) / K / 1e3
    # per head: Q K^T and S V (2 n_q n_k d each) and (S V)^T (S V) (2 n_q d^2)
    flops = n_kv * (4.0 * n_q * n_k * 128 + 2.0 * n_q * 128 * 128)
    tf = flops / t / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except (OSError, KeyError, ValueError):
        peak, peak_kind = 1900.0, "fallback bf16"
    print(json.dumps({
        "metric": "score-weighted value covariance TFLOP/s (C_S = (S V)^T (S V) / N, 8 KV heads of one layer)",
        "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": VCALIB_WORKLOAD, "n_kv_heads": n_kv, "calibration_queries": n_q,
                   "calibration_keys": n_k, "d": 128, "l2_policy": "inputs 24 MB, L2-resident (compute-bound)"},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                     "kernel": "sv_rows_kernel + sv_covariance_kernel (oscar_value_covariance)",
                     "algorithmic_flops": flops, "peak_kind": peak_kind},
        "gpu_launches": 3 * n_kv * K, "clocks": clk}))


def main():
    args = _args()
    if args.cpu_baseline_worker:
        cpu_baseline_worker(args.reps)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload == CALIB_WORKLOAD:
        run_calibration(args)
        return
    if args.workload == VCALIB_WORKLOAD:
        run_value_calibration(args)
        return
    if args.workload != WORKLOAD["workload"]:
        run_extra(args)
        return
    run_gpu(args)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark: GDN tail-replay state rebuild on GB300 (one rank per GPU).

A step is one gdn_replay call over one layer's replay batch (default: one
3277-token tail, 16 q/k heads shared by 32 v heads, d_k = d_v = 128, bf16
inputs, fp32 state) with its inputs resident in HBM.  Prints one JSON line
(rank 0).  ``--impl reference`` times the fp64 CPU oracle on the host cores
instead, on a bounded sample of the same workload.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launch stream; a 256 MiB memset flushes L2 between steps (outside the
events); a barrier and a device synchronize bracket the whole timed loop;
the reported time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN tail-replay tokens/s per layer; state-rebuild us @3.2K tail; % roofline"
CHUNK = 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="layer_r3277",
                    choices=["layer_r3277", "layer_r1638", "varlen", "full_32k", "tiny"])
    ap.add_argument("--precise", action="store_true", help="bf16 inputs on the fp32 CUDA-core path")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-depth", type=int, default=3, help="streams and buffer sets in the host-buffer pipeline")
    ap.add_argument("--no-rows", action="store_true", help="skip the varlen / full / chunk-operator / compose rows")
    ap.add_argument("--case", choices=["compose", "chunk_operator", "state_only"], default=None,
                    help="time one secondary workload alone and exit (16 x 2048 fp32 chunks at 32 heads, or "
                         "the 3277-token layer state only); the short command the kernel profiles are taken with")
    return ap.parse_args()


# ----------------------------------------------------------------------------- workload

def make_inputs(name: str, layer: int = 0):
    from gated_deltanet_state_chunked_gb300 import synthetic
    if name == "varlen":
        return synthetic.varlen_workload_inputs(layer)
    return synthetic.workload_inputs(name, layer)


def describe(name, x):
    lens = np.diff(x.cu_seqlens)
    return {
        "workload": name,
        "tails": int(x.n_seqs), "tokens": int(x.total_tokens),
        "tail_len_min": int(lens.min()) if len(lens) else 0, "tail_len_max": int(lens.max()) if len(lens) else 0,
        "h_k": x.h_k, "h_v": x.h_v, "d_k": x.d_k, "d_v": x.d_v,
        "inputs": x.dtype, "state": "f32", "S0": "zero", "chunk": CHUNK,
        "l2_flush": "256 MiB memset between timed steps",
    }


def algorithmic(x, with_O=True):
    """Algorithmic FLOPs and HBM bytes of one replay launch (fixed formulas)."""
    T, Hk, Hv, dk, dv, N = x.total_tokens, x.h_k, x.h_v, x.d_k, x.d_v, x.n_seqs
    e = 2 if x.dtype == "bf16" else 4
    flops = T * Hv * (6 * dk * dv + CHUNK * (6 * dk + 4 * dv))
    per_tok = 2 * Hk * dk * e + Hv * dv * e + 8 * Hv + (Hv * dv * e if with_O else 0)
    byts = T * per_tok + N * Hv * dv * dk * 4 + 4 * (N + 1)
    return flops, byts


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_state_chunked_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(f.encode())
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    for line in open(p):
        m = re.match(r"\s*traffic\s+workload=(\S+)\s+sources=(\w+)\s+bytes_per_launch=(\d+)", line)
        if m and m.group(1) == workload and m.group(2) == source_digest():
            return int(m.group(3))
    return None


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value over all ranks (the slowest rank's time); x itself on one rank."""
    if dist is None or not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [s.strip() for s in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ----------------------------------------------------------------------------- CPU oracle timing

def time_oracle(x, budget_s: float, max_reps: int = 50):
    """Time the fp64 oracle on a bounded sample of one layer's replay batch:
    whole (tail, head) problems, as many as fit in about budget_s.  Returns
    (tokens/s per layer, seconds, threads, sample description)."""
    import oracle
    pairs = [(s, h) for s in range(x.n_seqs) for h in range(x.h_v)]
    lens = np.diff(x.cu_seqlens)
    threads = oracle.num_threads()
    # probe with one problem per thread to estimate the rate
    probe = pairs[: max(1, min(len(pairs), threads))]
    t0 = time.perf_counter()
    oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, want_O=True, sel=probe)
    dt = time.perf_counter() - t0
    per_pair = dt / len(probe) * min(threads, len(probe))  # wall time per problem-wave slot
    n_fit = int(max(1, budget_s / max(per_pair, 1e-6) * threads))
    sample = pairs[: min(len(pairs), n_fit)]
    reps, total, t_start = 0, 0.0, time.perf_counter()
    while reps < max_reps:
        t0 = time.perf_counter()
        oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, want_O=True, sel=sample)
        total += time.perf_counter() - t0
        reps += 1
        if time.perf_counter() - t_start >= budget_s * 0.5 or len(sample) < len(pairs):
            break
    head_tokens = sum(int(lens[s]) for s, _ in sample) * reps
    tokens_per_layer = head_tokens / x.h_v  # a layer's token covers h_v heads
    desc = (f"{len(sample)} of {len(pairs)} (tail, v-head) replays x {reps} rep(s), full fp64 token loop "
            f"with outputs; tokens/s per layer = tail tokens x heads sampled / h_v / time")
    return tokens_per_layer / total, total, threads, desc


# ----------------------------------------------------------------------------- runs

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = make_inputs(args.workload)
    steps = []
    for i in range(args.warmup + args.steps):
        v, secs, threads, desc = time_oracle(x, budget_s=3.0, max_reps=1)
        if i >= args.warmup:
            steps.append((v, secs))
    value = statistics.mean(v for v, _ in steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(s for _, s in steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(args.workload, x),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _timed_us(fn, flush, reps, warmup=2):
    """Median device time of fn() in microseconds, L2 flushed before every call."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return float(np.median(ts))


def measure_rows(dev, flush, peaks, replay_us):
    """The other measured workloads: the varlen layer, the full 32K prefix against its 10% tail,
    and the chunk operators and composition of 16 isolated 2048-token chunks."""
    import torch

    from gated_deltanet_state_chunked_gb300 import api, synthetic
    import oracle

    def dev_inputs(x):
        dt = torch.bfloat16 if x.dtype == "bf16" else torch.float32
        f = lambda a, d: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(d)
        return dict(q=f(x.q, dt), k=f(x.k, dt), v=f(x.v, dt), g=f(x.g, torch.float32),
                    beta=f(x.beta, torch.float32), cu=f(x.cu_seqlens, torch.int32))

    rows = {}
    hbm = peaks["hbm_gbs"]
    # varlen layer: 64 tails of one layer
    x = synthetic.varlen_workload_inputs(0)
    d = dev_inputs(x)
    O = torch.empty((x.total_tokens, x.h_v, x.d_v), dtype=torch.bfloat16, device=dev)
    S = torch.empty((x.n_seqs, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
    us = _timed_us(lambda: api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], O_out=O, S_out=S),
                   flush, 5)
    fl, by = algorithmic(x, with_O=True)
    rows["varlen_layer"] = {"tails": x.n_seqs, "tokens": x.total_tokens, "us": us,
                            "tokens_per_s": x.total_tokens / (us * 1e-6), "hbm_frac": by / (us * 1e-6) / 1e9 / hbm,
                            "algorithmic_bytes": by, "algorithmic_flops": fl}
    del d, O, S
    # full 32K prefix vs its last 3277 tokens replayed from a zero state (config gates, then weak decay)
    for tag, gs in (("full_32k", 0.1), ("full_32k_weak_decay", 1e-3)):
        x = synthetic.workload_inputs("full_32k", gate_scale=gs)
        d = dev_inputs(x)
        S_full = torch.empty((1, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
        S_tail = torch.empty_like(S_full)
        r = 3277
        cu_tail = torch.tensor([0, r], dtype=torch.int32, device=dev)
        tail = {n: d[n][-r:].contiguous() for n in ("q", "k", "v", "g", "beta")}
        full_fn = lambda: api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], S_out=S_full,
                                         state_only=True)
        tail_fn = lambda: api.gdn_replay(tail["q"], tail["k"], tail["v"], tail["g"], tail["beta"], cu_tail,
                                         S_out=S_tail, state_only=True)
        full_us = _timed_us(full_fn, flush, 3) if tag == "full_32k" else None
        full_fn()
        tail_fn()
        torch.cuda.synchronize()
        err = oracle.rel_err(S_tail.double().cpu().numpy(), S_full.double().cpu().numpy())
        ent = {"replay_vs_full_rel_err_S": err, "tail_tokens": r, "gate_scale": gs}
        if full_us is not None:
            ent |= {"full_us_state_only": full_us, "replay_us_with_outputs": replay_us,
                    "speedup_full_over_replay": full_us / replay_us}
        rows[tag] = ent
        del d, tail
    # TF32 tensor peak of this GPU (a cuBLAS TF32 matmul, 8192^3, best of 5): the denominator for
    # the fp32-accurate contractions below, which run as three tf32 products each
    a32 = torch.randn((8192, 8192), dtype=torch.float32, device=dev)
    b32 = torch.randn((8192, 8192), dtype=torch.float32, device=dev)
    prev_tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    tts = []
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a32, b32)
        e1.record()
        torch.cuda.synchronize()
        tts.append(e0.elapsed_time(e1) * 1e-3)
    torch.backends.cuda.matmul.allow_tf32 = prev_tf32
    tf32_peak = 2 * 8192 ** 3 / min(tts[1:]) / 1e12
    del a32, b32
    rows["tf32_peak"] = {"tflops": tf32_peak, "how": "torch.matmul fp32 8192^3 with TF32 allowed (cuBLAS), best of 5"}
    # chunk operators of 16 x 2048 fp32 chunks and their composition (K = 16, 32 heads, d = 128)
    x = synthetic.chunk_workload_inputs()
    d = dev_inputs(x)
    K = x.n_seqs
    T = torch.empty((K, x.h_v, x.d_k, x.d_k), dtype=torch.float32, device=dev)
    Sl = torch.empty((K, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
    us = _timed_us(lambda: api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], d["cu"], T_out=T, Slocal_out=Sl),
                   flush, 2, warmup=1)
    rows_aug = x.d_v + x.d_k
    fl = x.total_tokens * x.h_v * (6 * x.d_k * rows_aug + 64 * (6 * x.d_k + 4 * rows_aug))
    rows["chunk_operator"] = {"chunks": K, "chunk_tokens": 2048, "heads": x.h_v, "dtype": "f32", "us": us,
                              "algorithmic_flops": fl, "tflops": fl / (us * 1e-6) / 1e12,
                              "frac_of_tf32_peak": fl / (us * 1e-6) / 1e12 / tf32_peak,
                              "path": "fp32 inputs: prep (norms, gates, Gram on warp-level split tf32, (I + A)^-1) "
                                      "into records, then the augmented-state scan [S; P] on tcgen05 in split tf32"}
    Tl, Sll = [T[j] for j in range(K)], [Sl[j] for j in range(K)]
    SK = torch.empty((x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
    us = _timed_us(lambda: api.gdn_compose(Tl, Sll, None, S_out=SK), flush, 10)
    by = K * x.h_v * (x.d_k * x.d_k + x.d_v * x.d_k) * 4 + x.h_v * x.d_v * x.d_k * 4
    fl = K * x.h_v * 2 * x.d_v * x.d_k * x.d_k
    rows["compose"] = {"K": K, "heads": x.h_v, "d": x.d_k, "us": us, "algorithmic_bytes": by,
                       "gbs": by / (us * 1e-6) / 1e9, "hbm_frac": by / (us * 1e-6) / 1e9 / hbm,
                       "algorithmic_flops": fl, "frac_of_tf32_peak": fl / (us * 1e-6) / 1e12 / tf32_peak,
                       "path": "operators in one array: tensor copies multicast over a 4-CTA cluster per head, "
                               "tcgen05 split tf32 (fp32 accuracy)" if x.d_k == 128 and x.d_v == 128
                       else "fp32 CUDA cores"}
    # the same composition with the operators at no common stride (the row-copy kernel)
    big = torch.empty((K + 2,) + tuple(T.shape[1:]), dtype=torch.float32, device=dev)
    slots = [K - j + (1 if j == 0 else 0) for j in range(K)]  # reversed, the first a slot further out
    for j in range(K):
        big[slots[j]].copy_(T[j])
    Tsc = [big[slots[j]] for j in range(K)]
    SK2 = torch.empty_like(SK)
    us2 = _timed_us(lambda: api.gdn_compose(Tsc, Sll, None, S_out=SK2), flush, 10)
    torch.cuda.synchronize()
    rows["compose_scattered"] = {"K": K, "heads": x.h_v, "d": x.d_k, "us": us2, "algorithmic_bytes": by,
                                 "gbs": by / (us2 * 1e-6) / 1e9, "hbm_frac": by / (us2 * 1e-6) / 1e9 / hbm,
                                 "path": "operators at no common stride: T rows by bulk copies, tcgen05 split tf32"}
    del big, Tsc
    api.gdn_get_status()
    rows |= measure_more_rows(dev, flush, peaks, dev_inputs)
    return rows


def measure_more_rows(dev, flush, peaks, dev_inputs):
    """Short tail and tiny workloads, all 48 varlen layers, the replay-error curve over the replay
    ratio, copy-stream overlap with a synthetic FA KV upload, and the last-block initializer."""
    import torch

    from gated_deltanet_state_chunked_gb300 import api, synthetic
    import oracle

    rows = {}
    hbm, bf16 = peaks["hbm_gbs"], peaks["bf16_tflops"]

    def replay_row(name, state_only=False, reps=10):
        x = synthetic.workload_inputs(name)
        d = dev_inputs(x)
        dt = torch.bfloat16 if x.dtype == "bf16" else torch.float32
        O = None if state_only else torch.empty((x.total_tokens, x.h_v, x.d_v), dtype=dt, device=dev)
        S = torch.empty((x.n_seqs, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
        us = _timed_us(lambda: api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], O_out=O, S_out=S,
                                              state_only=state_only), flush, reps)
        fl, by = algorithmic(x, with_O=not state_only)
        S_ref, _ = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, want_O=False,
                                 sel=[(0, 0), (0, x.h_v - 1)])
        Sh = S.double().cpu().numpy()
        err = max(oracle.rel_err(Sh[0, h], S_ref[0, h]) for h in (0, x.h_v - 1))
        return {"tokens": x.total_tokens, "heads": x.h_v, "d": x.d_k, "dtype": x.dtype, "state_only": state_only,
                "us": us, "tokens_per_s": x.total_tokens / (us * 1e-6), "algorithmic_bytes": by,
                "algorithmic_flops": fl, "hbm_frac": by / (us * 1e-6) / 1e9 / hbm,
                "tensor_frac": fl / (us * 1e-6) / 1e12 / bf16, "rel_err_S_sampled": err}

    rows["layer_r1638"] = replay_row("layer_r1638")
    rows["layer_r1638_state_only"] = replay_row("layer_r1638", state_only=True)
    rows["layer_r3277_state_only"] = replay_row("layer_r3277", state_only=True)
    rows["tiny"] = replay_row("tiny", reps=20)

    # 48 stacked independent layers of 64 concurrent tails: each layer its own tail lengths (from
    # the seed, as in the tests) and its own inputs, drawn on the GPU with the same distributions
    # (generating 48 x 1.6 GB on the host would take minutes); one call per layer, each timed.
    lay_us, lay_tok = [], []
    g = torch.Generator(device=dev)
    for layer in range(48):
        seed = synthetic.config_seed(2, layer)
        lens = synthetic.varlen_tail_lengths(64, seed)
        T = int(sum(lens))
        g.manual_seed(seed)
        unit = lambda shape: torch.nn.functional.normalize(torch.randn(shape, generator=g, device=dev), dim=-1)
        q, k = unit((T, 16, 128)).to(torch.bfloat16), unit((T, 16, 128)).to(torch.bfloat16)
        v = torch.randn((T, 32, 128), generator=g, device=dev).to(torch.bfloat16)
        beta = torch.sigmoid(torch.randn((T, 32), generator=g, device=dev))
        gg = -torch.nn.functional.softplus(torch.randn((T, 32), generator=g, device=dev) + 2.0) * 0.1
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device=dev)
        O = torch.empty((T, 32, 128), dtype=torch.bfloat16, device=dev)
        S = torch.empty((64, 32, 128, 128), dtype=torch.float32, device=dev)
        lay_us.append(_timed_us(lambda: api.gdn_replay(q, k, v, gg, beta, cu, O_out=O, S_out=S), flush, 2, warmup=1))
        lay_tok.append(T)
        del q, k, v, beta, gg, O, S
    tot_us = float(sum(lay_us))
    rows["varlen_48_layers"] = {"layers": 48, "tails_per_layer": 64, "tokens_total": int(sum(lay_tok)),
                                "us_total": tot_us, "us_per_layer_mean": tot_us / 48,
                                "us_per_layer_min": float(min(lay_us)), "us_per_layer_max": float(max(lay_us)),
                                "tokens_per_s_per_layer": float(sum(lay_tok)) / (tot_us * 1e-6),
                                "inputs": "values drawn on the GPU (torch.Generator, seeded per layer) with the "
                                          "workload's distributions; tail lengths from the seed"}

    # replay error against the full-prefix state over the replay ratio (32K prefix; weak-decay
    # gates make the dropped prefix state matter, the workload gates make it vanish)
    curve = {}
    for tag, gs in (("weak_decay", 1e-3), ("workload_gates", 0.1)):
        x = synthetic.workload_inputs("full_32k", gate_scale=gs)
        d = dev_inputs(x)
        S_full = torch.empty((1, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
        api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], S_out=S_full, state_only=True)
        pts = []
        for rho in (0.01, 0.02, 0.05, 0.10, 0.20):
            r = synthetic.tail_length(x.total_tokens, rho)
            tail = {n: d[n][-r:].contiguous() for n in ("q", "k", "v", "g", "beta")}
            S_t = torch.empty_like(S_full)
            api.gdn_replay(tail["q"], tail["k"], tail["v"], tail["g"], tail["beta"],
                           torch.tensor([0, r], dtype=torch.int32, device=dev), S_out=S_t, state_only=True)
            torch.cuda.synchronize()
            pts.append({"rho": rho, "tail_tokens": r,
                        "rel_err_S": oracle.rel_err(S_t.double().cpu().numpy(), S_full.double().cpu().numpy())})
        curve[tag] = pts
        del d
    rows["replay_error_vs_rho"] = {"prefix_tokens": 32768, "points": curve}

    # copy-stream overlap: a synthetic FA KV upload of the matched prefix (one full-attention
    # layer: 32768 tokens x 8 KV heads x 128 x (K, V), bf16 = 128 MiB) from pinned host memory,
    # serialised with one GDN layer's replay on one stream, then on a second stream beside it.
    x = synthetic.workload_inputs("layer_r3277")
    d = dev_inputs(x)
    O = torch.empty((x.total_tokens, x.h_v, x.d_v), dtype=torch.bfloat16, device=dev)
    S = torch.empty((1, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
    kv_bytes = 32768 * 8 * 128 * 2 * 2
    h_kv = torch.empty(kv_bytes, dtype=torch.uint8).pin_memory()
    d_kv = torch.empty(kv_bytes, dtype=torch.uint8, device=dev)
    s_main, s_copy = torch.cuda.current_stream(dev), torch.cuda.Stream(dev)
    replay = lambda st: api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], O_out=O, S_out=S, stream=st)

    def timed(fn, reps=5):
        ts = []
        for _ in range(reps + 1):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_main)
            fn()
            e1.record(s_main)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1) * 1e3)
        return float(np.median(ts[1:]))

    def copy_only():
        d_kv.copy_(h_kv, non_blocking=True)

    def serialised():
        d_kv.copy_(h_kv, non_blocking=True)
        replay(s_main)

    def overlapped():
        ev = torch.cuda.Event()
        ev.record(s_main)
        s_copy.wait_event(ev)
        with torch.cuda.stream(s_copy):
            d_kv.copy_(h_kv, non_blocking=True)
        replay(s_main)
        done = torch.cuda.Event()
        done.record(s_copy)
        s_main.wait_event(done)

    # the host link alone: the same bytes read back, and one copy each way at the same time (two
    # streams), the rates the end-to-end leg's uploads and read-backs share
    h_back = torch.empty(kv_bytes, dtype=torch.uint8).pin_memory()

    def read_back():
        h_back.copy_(d_kv, non_blocking=True)

    def both_ways():
        ev = torch.cuda.Event()
        ev.record(s_main)
        s_copy.wait_event(ev)
        with torch.cuda.stream(s_copy):
            h_back.copy_(d_kv, non_blocking=True)
        d_kv.copy_(h_kv, non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_copy)
        s_main.wait_event(done)

    t_copy, t_rep = timed(copy_only), timed(lambda: replay(s_main))
    t_ser, t_ovl = timed(serialised), timed(overlapped)
    t_back, t_both = timed(read_back), timed(both_ways)
    rows["copy_overlap"] = {"fa_kv_bytes": kv_bytes, "copy_us": t_copy, "replay_us": t_rep,
                            "serialised_us": t_ser, "overlapped_us": t_ovl,
                            "hidden_us": t_copy + t_rep - t_ovl, "h2d_gbs": kv_bytes / (t_copy * 1e-6) / 1e9,
                            "d2h_gbs": kv_bytes / (t_back * 1e-6) / 1e9,
                            "both_ways_gbs": 2 * kv_bytes / (t_both * 1e-6) / 1e9,
                            "fa_kv": "one full-attention layer: 32768 tokens x 8 KV heads x 128 x (K, V), bf16, pinned host"}
    del h_kv, d_kv, d, h_back

    # LinearKV's last-block initializer (the last chunk's local state alone) against the exact
    # composition of all chunk operators and against sequential replay of all chunks, on 16
    # isolated 2048-token chunks (workload gates, then weak decay)
    lb = {}
    for fam, scalar in (("gdn", False), ("scalar_decay", True)):
        for tag, wd in (("workload_gates", False), ("weak_decay", True)):
            x = synthetic.chunk_workload_inputs(weak_decay=wd)
            d = dev_inputs(x)
            K = x.n_seqs
            T = torch.empty((K, x.h_v, x.d_k, x.d_k), dtype=torch.float32, device=dev)
            Sl = torch.empty((K, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
            api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], d["cu"], T_out=T, Slocal_out=Sl,
                                   scalar_decay=scalar)
            SK = api.gdn_compose([T[j] for j in range(K)], [Sl[j] for j in range(K)])
            S_seq = torch.empty((1, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
            cu_all = torch.tensor([0, x.total_tokens], dtype=torch.int32, device=dev)
            api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_all, S_out=S_seq, state_only=True,
                           precise=True, scalar_decay=scalar)
            torch.cuda.synchronize()
            ref = S_seq[0].double().cpu().numpy()
            lb[f"{fam}_{tag}"] = {"exact_composition_rel_err": oracle.rel_err(SK.double().cpu().numpy(), ref),
                                  "last_block_rel_err": oracle.rel_err(Sl[K - 1].double().cpu().numpy(), ref)}
            del d
    rows["last_block_initializer"] = {"chunks": 16, "chunk_tokens": 2048, "heads": 32,
                                      "vs": "sequential replay of all chunks (fp32 path)",
                                      "families": "gdn: dense rank-1 transitions; scalar_decay: Mamba-2 scalar transitions",
                                      "cases": lb}

    # chunk-operator parallel scan: the 3277-token tail split into G segments whose operators are
    # built side by side (fp32 chunk-operator path), then composed, against the sequential replay
    x = synthetic.workload_inputs("layer_r3277")
    d = dev_inputs(x)
    S_seq = torch.empty((1, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
    seq_us = _timed_us(lambda: api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], S_out=S_seq,
                                              state_only=True), flush, 5)
    ps = {"sequential_state_only_us": seq_us, "segments": []}
    for G in (2, 4, 8):
        edges = [round(i * x.total_tokens / G) for i in range(G + 1)]
        cu_g = torch.tensor(edges, dtype=torch.int32, device=dev)
        T = torch.empty((G, x.h_v, x.d_k, x.d_k), dtype=torch.float32, device=dev)
        Sl = torch.empty((G, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
        SK = torch.empty((x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
        op = lambda: api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], cu_g, T_out=T, Slocal_out=Sl)
        comp = lambda: api.gdn_compose([T[j] for j in range(G)], [Sl[j] for j in range(G)], S_out=SK)
        op_us, comp_us = _timed_us(op, flush, 3, warmup=1), _timed_us(comp, flush, 5)
        torch.cuda.synchronize()
        ps["segments"].append({"G": G, "chunk_operators_us": op_us, "compose_us": comp_us, "total_us": op_us + comp_us,
                               "rel_err_vs_sequential": oracle.rel_err(SK.double().cpu().numpy(),
                                                                       S_seq[0].double().cpu().numpy())})
    rows["parallel_scan_replay"] = ps
    del d
    api.gdn_get_status()
    return rows


def run_ours(args):
    import torch
    import torch.distributed as dist

    from gated_deltanet_state_chunked_gb300 import _lib, api

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())
    _lib.load()
    x = make_inputs(args.workload, layer=rank)  # each rank replays its own layer's batch
    dt = torch.bfloat16 if x.dtype == "bf16" else torch.float32

    def dtens(a, d):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(d)

    q, k, v = dtens(x.q, dt), dtens(x.k, dt), dtens(x.v, dt)
    g, beta = dtens(x.g, torch.float32), dtens(x.beta, torch.float32)
    cu = dtens(x.cu_seqlens, torch.int32)
    T, n = x.total_tokens, x.n_seqs
    O = torch.empty((T, x.h_v, x.d_v), dtype=dt, device=dev)
    S = torch.empty((n, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.gdn_replay(q, k, v, g, beta, cu, None, O_out=O, S_out=S, precise=args.precise, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    api.gdn_get_status()

    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(dev.index)
    sampler = ClockSampler(gpu_id)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    tensor_path = x.dtype == "bf16" and not args.precise and x.d_k == 128 and x.d_v == 128
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    api.gdn_get_status()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    stages = None
    if tensor_path:
        # Per-kernel durations, after the timed region: a stage event recorded between the prep
        # and scan kernels (which makes the library run them one after the other instead of
        # overlapping the scan's start with the prep's last CTAs).
        ks = min(args.steps, 10)
        s0 = [torch.cuda.Event(enable_timing=True) for _ in range(ks)]
        mids = [torch.cuda.Event(enable_timing=True) for _ in range(ks)]
        s1 = [torch.cuda.Event(enable_timing=True) for _ in range(ks)]
        for e in mids:
            e.record(stream)  # create the event handles before handing them to the library
        for i in range(ks):
            flush.zero_()
            s0[i].record(stream)
            api.gdn_set_stage_event(mids[i])
            step()
            s1[i].record(stream)
        torch.cuda.synchronize(dev)
        api.gdn_get_status()
        prep_ms = sum(a.elapsed_time(m) for a, m in zip(s0, mids)) / ks
        scan_ms = sum(m.elapsed_time(b) for m, b in zip(mids, s1)) / ks
        stages = {"chunk_prep_kernel_us": prep_ms * 1e3, "chunk_scan_kernel_us": scan_ms * 1e3,
                  "dominant": "chunk_scan_kernel" if scan_ms >= prep_ms else "chunk_prep_kernel",
                  "measured": f"{ks} separate calls with the kernels serialised by a stage event"}
    ms = max_over_ranks(ms, dist, dev)

    # parity of the last timed step on a few sampled (tail, head) problems
    import oracle
    sel = [(0, 0), (0, x.h_v - 1), (x.n_seqs - 1, x.h_v // 2)] if rank == 0 else None
    parity = None
    if sel is not None:
        S_ref, O_ref = oracle.replay(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, want_O=True, sel=sel)
        Sh, Oh = S.cpu().double().numpy(), O.float().cpu().double().numpy()
        es = max(oracle.rel_err(Sh[s, h], S_ref[s, h]) for s, h in sel)
        rows = [(slice(int(x.cu_seqlens[s]), int(x.cu_seqlens[s + 1])), h) for s, h in sel]
        eo = max(oracle.rel_err(Oh[r, h], O_ref[r, h]) for r, h in rows)
        parity = {"rel_err_S_max": es, "rel_err_O_max": eo, "sampled": [list(p) for p in sel]}

    # end to end through the public call with host buffers: H2D inputs, replay, D2H result
    e2e = None
    if not args.no_e2e:
        # End to end through gdn_replay with host buffers: every step uploads its inputs from
        # pinned host memory, replays, and reads O and S back.  NB streams and device buffer
        # sets in rotation, so that later steps' uploads overlap a step's replay and read-back
        # (as a server would pipeline requests); the timed region spans all K steps.
        # Each step's inputs sit packed in one pinned host buffer and go up in one copy; O and S
        # come back in one copy as well (one large transfer per direction runs closer to the host
        # link's rate than several smaller ones).
        def packed(specs, device, pin):
            offs, total = [], 0
            for shape, dtype in specs:
                total = (total + 255) // 256 * 256
                offs.append(total)
                total += int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            buf = torch.empty(total, dtype=torch.uint8, device=device)
            if pin:
                buf = buf.pin_memory()
            views = [buf[o:o + int(np.prod(sh)) * torch.empty((), dtype=dty).element_size()].view(dty).view(sh)
                     for o, (sh, dty) in zip(offs, specs)]
            return buf, views

        in_specs = [(tuple(q.shape), dt), (tuple(k.shape), dt), (tuple(v.shape), dt), (tuple(g.shape), torch.float32),
                    (tuple(beta.shape), torch.float32), (tuple(cu.shape), torch.int32)]
        out_specs = [(tuple(O.shape), dt), (tuple(S.shape), torch.float32)]
        hin, hin_v = packed(in_specs, "cpu", True)
        for dst, a, dty in zip(hin_v, (x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens.astype(np.int32)),
                               (dt, dt, dt, torch.float32, torch.float32, torch.int32)):
            dst.copy_(torch.from_numpy(np.ascontiguousarray(a)).to(dty))
        NB = args.e2e_depth
        hout = [packed(out_specs, "cpu", True) for _ in range(NB)]
        dins = [packed(in_specs, dev, False) for _ in range(NB)]
        douts = [packed(out_specs, dev, False) for _ in range(NB)]
        streams = [stream] + [torch.cuda.Stream(dev) for _ in range(NB - 1)]
        h2d = hin.numel()  # bytes of the one upload (the tensors plus their alignment gaps)
        d2h = hout[0][0].numel()

        def e2e_step(i):
            b = i % NB
            st = streams[b]
            (dbuf, (dq, dk, dv, dg, db, dcu)), (obuf, (dO, dS)) = dins[b], douts[b]
            with torch.cuda.stream(st):
                dbuf.copy_(hin, non_blocking=True)
                api.gdn_replay(dq, dk, dv, dg, db, dcu, None, O_out=dO, S_out=dS, precise=args.precise, stream=st)
                hout[b][0].copy_(obuf, non_blocking=True)

        def e2e_run(n):
            t0, t1, j1 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            t0.record(streams[0])
            for st in streams[1:]:
                st.wait_event(t0)
            for i in range(n):
                e2e_step(i)
            for st in streams[1:]:
                j = torch.cuda.Event()
                j.record(st)
                streams[0].wait_event(j)
            t1.record(streams[0])
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1)

        e2e_run(max(2, args.warmup))
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        e2e_ms = e2e_run(args.steps) / args.steps
        api.gdn_get_status()
        e2e_ms = max_over_ranks(e2e_ms, dist, dev)
        # One call alone, not pipelined: upload, replay, read-back on one stream (the latency a
        # cache hit waits for when nothing else is in flight).
        def latency_once():
            (dbuf, (dq, dk, dv, dg, db, dcu)), (obuf, (dO, dS)) = dins[0], douts[0]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            dbuf.copy_(hin, non_blocking=True)
            api.gdn_replay(dq, dk, dv, dg, db, dcu, None, O_out=dO, S_out=dS, precise=args.precise, stream=stream)
            hout[0][0].copy_(obuf, non_blocking=True)
            t1.record(stream)
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1)

        for _ in range(3):
            latency_once()
        lat_ms = float(np.median([latency_once() for _ in range(max(5, args.steps))]))
        api.gdn_get_status()
        e2e = {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelining": f"{NB} streams, {NB} buffer sets: uploads of later steps overlap a step's replay and read-back; one copy per direction per step",
               "latency_ms_one_call": lat_ms,
               "latency": "one call alone on one stream: one upload of the packed inputs from pinned memory, the replay, one read-back of O and S"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v_cpu, secs, threads, desc = time_oracle(x, budget_s=15.0)
        cpu = {"value": v_cpu, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": secs}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    flops, byts = algorithmic(x, with_O=True)
    peaks, peak_src = load_peaks()
    rows = None
    if world == 1 and not args.no_rows:
        rows = measure_rows(dev, flush, peaks, ms * 1e3)
    t_s = ms * 1e-3
    gbs = byts / t_s / 1e9
    tfs = flops / t_s / 1e12
    traffic = recorded_traffic(args.workload)
    roofline = {
        "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
        "traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
        else "fallback 6.8 TB/s",
        "kernel": "gdn_replay call = chunk_prep_kernel + chunk_scan_kernel (one launch of the path)",
        "stages": stages, "algorithmic_bytes": byts, "algorithmic_flops": flops,
        "tensor": {"achieved": tfs, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": tfs / peaks["bf16_tflops"]},
    }
    line = {
        "metric": METRIC, "value": world * T / t_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "state_rebuild_us": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": x.dtype, "data": "synthetic",
        "config": describe(args.workload, x) | {"path": "precise" if args.precise else "default",
                                                "parallelism": f"replicas x{world}"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        # per call: the two chunk kernels, plus the tail-order kernel when several tails share a call
        "gpu_launches": args.steps * (2 + (1 if tensor_path and x.n_seqs > 1 else 0)),
        "clocks": clocks, "parity": parity, "rows": rows,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_case(args):
    """One secondary workload alone: the chunk operators of 16 isolated 2048-token fp32 chunks
    (32 heads, d = 128), their composition (K = 16 operators in one array), or the 3277-token
    layer replayed state only, each timed over a few calls with the L2 flushed before every call."""
    import torch
    from gated_deltanet_state_chunked_gb300 import _lib, api, synthetic
    _lib.load(build=True)
    dev = torch.device("cuda", 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    if args.case == "state_only":
        x = make_inputs("layer_r3277")
        f = lambda a, t: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(t)  # noqa: E731
        d = dict(q=f(x.q, torch.bfloat16), k=f(x.k, torch.bfloat16), v=f(x.v, torch.bfloat16),
                 g=f(x.g, torch.float32), beta=f(x.beta, torch.float32), cu=f(x.cu_seqlens, torch.int32))
        S = torch.empty((x.n_seqs, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
        rep = lambda: api.gdn_replay(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], S_out=S, state_only=True)
        us = _timed_us(rep, flush, max(args.steps, 1), warmup=max(args.warmup, 1))
        api.gdn_get_status()
        print(json.dumps({"case": args.case, "us": us, "steps": args.steps, "warmup": args.warmup}))
        return
    x = synthetic.chunk_workload_inputs()
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(x, k))).to(dev) for k in ("k", "v", "g", "beta")}
    d["cu"] = torch.from_numpy(np.ascontiguousarray(x.cu_seqlens, dtype=np.int32)).to(dev)
    K = x.n_seqs
    T = torch.empty((K, x.h_v, x.d_k, x.d_k), dtype=torch.float32, device=dev)
    Sl = torch.empty((K, x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
    op = lambda: api.gdn_chunk_operator(d["k"], d["g"], d["beta"], d["v"], d["cu"], T_out=T, Slocal_out=Sl)
    if args.case == "chunk_operator":
        us = _timed_us(op, flush, max(args.steps, 1), warmup=max(args.warmup, 1))
    else:
        op()
        SK = torch.empty((x.h_v, x.d_v, x.d_k), dtype=torch.float32, device=dev)
        Tl, Sll = [T[j] for j in range(K)], [Sl[j] for j in range(K)]
        us = _timed_us(lambda: api.gdn_compose(Tl, Sll, None, S_out=SK), flush, max(args.steps, 1),
                       warmup=max(args.warmup, 1))
    api.gdn_get_status()
    print(json.dumps({"case": args.case, "us": us, "steps": args.steps, "warmup": args.warmup}))


def main():
    args = parse_args()
    if args.case:
        run_case(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Throughput benchmark of the low-bit decode GEMV hot path on GB300.

One step = one decode pass over a Llama-3-8B-shaped layer through every row of
the hot path:
  * the 7 linears in Group-32 asymmetric 4-bit (q, k, v, o, gate, up, down), M = 1;
  * the same 7 linears in 2-bit Lloyd-Max codebook with the top 3.5 % profile-
    guided FP16 outlier columns, M = 1;
  * the 4-bit gate and down projections as a small-M batch (M = 4).
Inputs are seeded synthetic data with the shapes and distributions of the
decode configurations (see bit_weight_only_lbq_gb300/synth.py).  The packed
weights of a step (291 MB) are held in 3 rotating replicas, so consecutive steps
never find their weights in the 126 MB L2.

A step is three grouped launches, one per row of the path, each a fused sweep
over its matrices (lbq_gemv_grouped): the 4-bit layer sweep, the 2-bit layer
sweep and the small-M batch.  The step is captured once per replica as a CUDA
graph (the three launches chained with programmatic dependent launch) and
timed with CUDA events around K replays.  Each grouped launch is then timed on
its own (rotating copies, >= 512 MB per pass) for the roofline figure, and each
of the 16 matrices alone for the per-call table.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 run under torch.distributed.run: every rank runs an independent
replica (the path has no exchange step) and rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_weight_only_lbq_gb300 import synth  # noqa: E402

REPLICAS = 3
SMALL_M = 4
SAMPLE_ROWS_MAX = 1024
L2_ROTATION_BYTES = 512 << 20  # distinct weight bytes one timing pass rotates through (4x L2)
# DRAM bytes (read + write) per grouped launch from ncu captures of the same
# launches (profiles/); valid only for the kernel source they were taken on.
TRAFFIC_CAPTURE = {"kernel_sha256_prefix": "22be62a830ce8505",
                   "traffic": {"w4_layer_sweep": 129267712, "w2_layer_sweep": 100116736,
                               "w4_smallM_gate_down": 68175872}}
METRIC = "W4/W2 decode GEMV µs/call and HBM GB/s (% of GB300 roofline); implied tokens/s"
W4_BYTES_PER_WEIGHT = 0.578125      # 4 bits + FP16 scale / 32 + 4-bit zero / 32
W2_BYTES_PER_WEIGHT = 0.375         # 2 bits + FP16 S / 32 + FP16 Z / 32


def algorithmic_bytes(kind: str, N: int, K: int, n_out: int, M: int = 1) -> int:
    """Bytes a launch must move at minimum: packed weights, group metadata,
    outlier indices and values, the activations read and the outputs written."""
    per_w = W4_BYTES_PER_WEIGHT if kind == "w4" else W2_BYTES_PER_WEIGHT
    return int(per_w * N * K + n_out * (4 + 2 * N) + 2 * K * M + 2 * N * M)


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest of every rank's value (each rank calls it); the value itself
    on one process.  Timings are reduced this way: the job takes as long as its
    slowest rank."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes: int, world: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: the bytes all ranks streamed (each rank runs its own
    replica of the step) over the slowest rank's time."""
    return step_bytes * world * steps / seconds / 1e9


def kernel_source_hash() -> str:
    import hashlib
    src = os.path.join(ROOT, "bit_weight_only_lbq_gb300", "csrc", "lbq_gemv.cu")
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples every 200 ms while the benchmark runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def wait_first(self, timeout: float = 5.0):
        """Block until the sampler has produced its first line (or timeout)."""
        t = time.time()
        while self.proc is not None and not self.samples and time.time() - t < timeout:
            time.sleep(0.02)

    def summary(self, t0: float, t1: float, w0: float = None, w1: float = None) -> dict:
        """Clock record of the timed region [t0, t1] and of the measurement window
        [w0, w1] around it (warm-up, timed region and the per-launch timing passes,
        all under the same load).  The median and the reasons come from the window
        when the timed region is too short to hold a 200 ms sample."""
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        window = [s for t, s in self.samples if (w0 if w0 is not None else t0) <= t <= (w1 if w1 is not None else t1)]
        used = inside if inside else (window if window else [s for _, s in self.samples[-3:]])
        sm = [float(s[1]) for s in used if len(s) > 8 and s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in used if len(s) > 8 and s[2].replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in used:
            if len(s) > 8:
                for i, n in enumerate(names):
                    if s[5 + i].lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples_in_region": len(inside), "samples_in_window": len(window),
                "source": "timed region" if inside else "measurement window (warm-up, timed steps, per-launch "
                                                         "timing passes)"}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def make_workload(lbq, rank: int):
    """Pack the step's 16 matrices on the host (C++ packers) and return host data."""
    layer = []
    for li, (name, N, K) in enumerate(synth.LLAMA3_8B_LINEARS):
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W4, layer_id=li + 100 * rank)
        x = synth.activations(1, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)[0]
        layer.append(dict(kind="w4", name=name, N=N, K=K, n_out=0, M=1, blob=lbq.pack_w4(W), x=x,
                          W_head=W[:SAMPLE_ROWS_MAX].copy(), idx=np.zeros(0, np.int32), li=li + 100 * rank))
    for li, (name, N, K) in enumerate(synth.LLAMA3_8B_LINEARS):
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W2, layer_id=li + 100 * rank)
        prof = synth.profile_vectors(K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
        idx = lbq.select_outliers_impact(W, prof, 0.035)
        x = synth.activations(1, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)[0]
        layer.append(dict(kind="w2", name=name, N=N, K=K, n_out=len(idx), M=1, blob=lbq.pack_w2cb(W, idx), x=x,
                          W_head=W[:SAMPLE_ROWS_MAX].copy(), idx=idx))
    for li in (4, 6):
        name, N, K = synth.LLAMA3_8B_LINEARS[li]
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_SMALL_M, layer_id=li + 100 * rank)
        X = synth.activations(SMALL_M, K, workload=synth.WL_SMALL_M, layer_id=li)
        layer.append(dict(kind="w4m", name=name, N=N, K=K, n_out=0, M=SMALL_M, blob=lbq.pack_w4(W), x=X,
                          W_head=W[:SAMPLE_ROWS_MAX].copy(), idx=np.zeros(0, np.int32)))
    for e in layer:
        e["bytes"] = algorithmic_bytes("w4" if e["kind"] != "w2" else "w2", e["N"], e["K"], e["n_out"], e["M"])
    return layer


def reps_i(reps, i):
    return [reps[r][i] for r in range(len(reps))]


GROUPS = (("w4_layer_sweep", "w4"), ("w2_layer_sweep", "w2"), ("w4_smallM_gate_down", "w4m"))


def group_members(layer, kind):
    return [i for i, e in enumerate(layer) if e["kind"] == kind]


def group_args(lbq, layer, members, blobs, xs, ys):
    """Problem tuples of a grouped launch; blobs/xs/ys indexed like layer."""
    probs = []
    for i in members:
        e = layer[i]
        probs.append((blobs[i], e["N"], e["K"], e["n_out"], xs[i], e["K"], ys[i], e["N"]))
    return probs


def launch_group(lbq, layer, kind, blobs, xs, ys, pdl):
    members = group_members(layer, kind)
    lk = lbq.LBQ_KIND_W2CB if kind == "w2" else lbq.LBQ_KIND_W4
    M = layer[members[0]]["M"]
    lbq.gemv_grouped(lk, group_args(lbq, layer, members, blobs, xs, ys), M=M, pdl=pdl)


def group_launch_count(lbq, layer, kind, blobs, xs, ys):
    members = group_members(layer, kind)
    lk = lbq.LBQ_KIND_W2CB if kind == "w2" else lbq.LBQ_KIND_W4
    return lbq.gemv_grouped_launches(lk, group_args(lbq, layer, members, blobs, xs, ys), M=layer[members[0]]["M"])


def launch(lbq, e, blob, x, y, pdl):
    M = e.get("M", 1)
    if e["kind"] == "w2" and M > 1:
        lbq.gemm_w2cb_outlier_smallM(blob, M, e["N"], e["K"], e["n_out"], x, e["K"], y, e["N"], pdl=pdl)
    elif e["kind"] == "w2":
        lbq.gemv_w2cb_outlier(blob, e["N"], e["K"], e["n_out"], x, y, pdl=pdl)
    elif e["kind"] == "w4" and M == 1:
        lbq.gemv_w4a16(blob, e["N"], e["K"], e["n_out"], x, y, pdl=pdl)
    else:
        lbq.gemm_w4a16_smallM(blob, M, e["N"], e["K"], e["n_out"], x, e["K"], y, e["N"], pdl=pdl)


# ---------------------------------------------------------------------------
# reference arm: the FP64 CPU oracle
# ---------------------------------------------------------------------------

def oracle_workload(rows: int):
    """The step's 16 matrices built with the oracle alone (no native code): the
    first `rows` rows of each seeded weight matrix, the 2-bit outlier columns
    chosen by the oracle's impact-score selection over the whole matrix, and the
    activations.  Entries as make_workload's, with W_head holding the rows."""
    from oracle import lbq_oracle as O
    layer = []
    for li, (name, N, K) in enumerate(synth.LLAMA3_8B_LINEARS):
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)
        layer.append(dict(kind="w4", name=name, N=N, K=K, n_out=0, M=1, W_head=W[:rows].copy(),
                          idx=np.zeros(0, np.int32), x=synth.activations(1, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)[0]))
    for li, (name, N, K) in enumerate(synth.LLAMA3_8B_LINEARS):
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
        idx = O.select_outliers_impact(W, synth.profile_vectors(K, workload=synth.WL_LLAMA8B_W2, layer_id=li))
        layer.append(dict(kind="w2", name=name, N=N, K=K, n_out=len(idx), M=1, W_head=W[:rows].copy(), idx=idx,
                          x=synth.activations(1, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)[0]))
    for li in (4, 6):
        name, N, K = synth.LLAMA3_8B_LINEARS[li]
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_SMALL_M, layer_id=li)
        layer.append(dict(kind="w4m", name=name, N=N, K=K, n_out=0, M=SMALL_M, W_head=W[:rows].copy(),
                          idx=np.zeros(0, np.int32), x=synth.activations(SMALL_M, K, workload=synth.WL_SMALL_M, layer_id=li)))
    return layer


def oracle_sample(layer, rows_per_matrix: int):
    """A step of the oracle over the first rows of every matrix of the step.  The
    oracle packs its own blob of those rows (untimed); the returned step times
    its FP64 dequantise-from-bytes + matvec and returns the algorithmic bytes."""
    from oracle import lbq_oracle as O
    prepared = []
    for e in layer:
        R = min(rows_per_matrix, e["N"], len(e["W_head"]))
        pack = O.pack_w2cb if e["kind"] == "w2" else O.pack_w4
        prepared.append((e, R, pack(e["W_head"][:R], e["idx"])))

    def step():
        nbytes = 0
        for e, R, blob in prepared:
            O.gemm(blob, e["x"])
            nbytes += algorithmic_bytes("w4" if e["kind"] != "w2" else "w2", R, e["K"], e["n_out"], e["M"])
        return nbytes
    return step, prepared


def oracle_figures(layer, rows: int, reps: int) -> dict:
    """The three CPU figures of the oracle over a row sample of the step (each
    scaled to GB/s of the sample's algorithmic bytes): (i) packing (quantise +
    pack, FP64), (ii) dequantise-from-bytes + matvec, (iii) matvec alone on the
    cached FP64 matrix the blob applies."""
    from oracle import lbq_oracle as O
    t = time.perf_counter()
    step, prepared = oracle_sample(layer, rows)
    t_pack = time.perf_counter() - t
    nbytes = step()
    t = time.perf_counter()
    for _ in range(reps):
        step()
    t_step = (time.perf_counter() - t) / reps
    cached = [(e, O.dequant_eff(blob), np.asarray(e["x"], np.float16).astype(np.float64)) for e, _, blob in prepared]
    t = time.perf_counter()
    for _ in range(reps):
        for e, Wh, x in cached:
            Wh @ x.T
    t_mv = (time.perf_counter() - t) / reps
    weights = sum(R * e["K"] for e, R, _ in prepared)
    return {"rows": rows, "bytes": nbytes, "weights": weights,
            "pack": {"s": round(t_pack, 4), "weights_per_s": round(weights / t_pack, 1)},
            "dequant_matvec": {"s": round(t_step, 5), "GB_s": round(nbytes / t_step / 1e9, 6)},
            "matvec_cached": {"s": round(t_mv, 5), "GB_s": round(nbytes / t_mv / 1e9, 6)}}


def oracle_70b_extrapolated(rows: int = 8) -> dict:
    """The Llama-3-70B decode weight sweep on the host: one sample of `rows` rows of each Llama-3-70B linear
    shape and of the lm_head, oracle dequantise-from-bytes + matvec, scaled by
    each shape's rows and count to one token's 80 x 7 + 1 matrices.  Extrapolated,
    never run whole (the oracle would hold 69.5 G FP64 weights)."""
    from oracle import lbq_oracle as O
    total = 0.0
    parts = []
    shapes = [(n, N, K, synth.LLAMA3_70B_LAYERS) for (n, N, K) in synth.LLAMA3_70B_LINEARS]
    hn, hN, hK = synth.LLAMA3_70B_LM_HEAD
    shapes.append((hn, hN, hK, 1))
    for name, N, K, count in shapes:
        W = synth.weights_heavy_cols(rows, K, workload=synth.WL_LLAMA70B, layer_id=len(parts))
        blob = O.pack_w4(W)
        x = synth.activations(1, K, workload=synth.WL_LLAMA70B, layer_id=K)[0]
        t = time.perf_counter()
        O.gemm(blob, x)
        dt = time.perf_counter() - t
        s_shape = dt / rows * N * count
        total += s_shape
        parts.append({"linear": name, "N": N, "K": K, "count": count, "s_per_token": round(s_shape, 3)})
    nbytes = sum(algorithmic_bytes("w4", N, K, 0) * c for (_, N, K, c) in shapes)
    return {"label": "extrapolated from %d-row samples" % rows, "s_per_token": round(total, 2),
            "GB_s": round(nbytes / total / 1e9, 6), "per_shape": parts}


def run_reference(args, rank, world):
    """The reference arm: the FP64 oracle as it stands, on the host cores, over a
    bounded row sample of the step, with inputs built by the oracle alone."""
    if rank != 0:
        return 0
    budget_s = 120.0
    rows = 64
    layer = oracle_workload(rows)
    step, _ = oracle_sample(layer, rows)
    t = time.perf_counter()
    step()
    one = time.perf_counter() - t
    per_step_budget = budget_s / max(1, args.steps + args.warmup)
    while rows > 1 and one > per_step_budget:
        rows //= 2
        step, _ = oracle_sample(layer, rows)
        t = time.perf_counter()
        step()
        one = time.perf_counter() - t
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += step()
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "first %d rows of each of the step's 16 matrices per step (FP64 NumPy "
                                   "dequantise-from-bytes + matvec; inputs and outlier columns from the oracle)"
                                   % rows},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict():
    return {"workload": "llama3_8b_layer_decode: 7 linears W4A16 G32 + 7 linears W2 Lloyd-Max G32 with "
                        "top-3.5% FP16 outliers + W4 gate/down small-M M=4, one token; each row "
                        "one fused sweep (grouped launch) over its matrices",
            "linears": [list(x) for x in synth.LLAMA3_8B_LINEARS], "small_m": SMALL_M,
            "l2": "inputs larger than L2: 3 rotating replicas of the 291 MB step",
            "parallelism": "replicas (one independent layer per GPU)"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="lbq", choices=["lbq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep70b", action="store_true", help="skip the Llama-3-70B weight sweep detail")
    ap.add_argument("--no-smallm-sweep", action="store_true", help="skip the small-M (M = 2..64) detail")
    ap.add_argument("--single", default=None,
                    help="kind:N:K:n_out:M - time one kernel configuration alone (profiling aid), "
                         "kind in w4, w2, w4m; sweep:KIND (one grouped launch of the step); "
                         "kv:ROWS:WIDTH (KV cache read); refine:N:K:k (select + apply); "
                         "embed:V:D:T (fused row gather of T token ids from a V x D 4-bit table)")
    args = ap.parse_args()
    if args.single:
        return run_single(args)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    from bit_weight_only_lbq_gb300 import lbq

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    layer = make_workload(lbq, rank)
    dev = torch.device("cuda", local_rank)
    step_bytes = sum(e["bytes"] for e in layer)

    # device buffers: REPLICAS copies of every blob, activations, outputs
    reps = []
    for r in range(REPLICAS):
        reps.append([torch.from_numpy(e["blob"]).to(dev) for e in layer])
    # the activations of all matrices in one device buffer, the outputs in another
    # (views of 16-byte aligned slices), so a step's inputs and results cross the
    # host link in one copy each
    x_all = torch.from_numpy(np.concatenate([np.ascontiguousarray(e["x"], dtype=np.float16).reshape(-1)
                                             for e in layer])).to(dev)
    y_all = torch.empty(sum(e["M"] * e["N"] for e in layer), dtype=torch.float16, device=dev)
    xs, ys, xo, yo = [], [], 0, 0
    for e in layer:
        n = int(np.asarray(e["x"]).size)
        xs.append(x_all[xo:xo + n].view(np.asarray(e["x"]).shape))
        ys.append(y_all[yo:yo + e["M"] * e["N"]].view(e["M"], e["N"]))
        assert (xo * 2) % 16 == 0 and (yo * 2) % 16 == 0
        xo += n
        yo += e["M"] * e["N"]
    launches_per_step = sum(group_launch_count(lbq, layer, kind, reps[0], xs, ys) for _, kind in GROUPS)

    def step_launches(blobs):
        for _, kind in GROUPS:
            launch_group(lbq, layer, kind, blobs, xs, ys, pdl=True)

    stream = torch.cuda.Stream(device=dev)
    graphs = []
    with torch.cuda.stream(stream):
        for r in range(REPLICAS):                      # eager warm-up (sets kernel attributes)
            step_launches(reps[r])
        stream.synchronize()
        assert lbq.device_error(stream) == 0
        for r in range(REPLICAS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step_launches(reps[r])
            graphs.append(g)

    clocks = ClockSampler(local_rank)
    clocks.start()
    clocks.wait_first()
    w_wall0 = time.time()
    with torch.cuda.stream(stream):
        # at least W warm-up steps, and at least 0.5 s of them, so the clocks have
        # settled under load and the sampler has seen it
        s = 0
        while s < max(3, args.warmup) or time.time() - w_wall0 < 0.5:
            graphs[s % REPLICAS].replay()
            s += 1
            if s % 200 == 0:
                stream.synchronize()
        stream.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        t_wall0 = time.time()
        ev0.record(stream)
        for s in range(args.steps):
            graphs[s % REPLICAS].replay()
        ev1.record(stream)
        ev1.synchronize()
        t_wall1 = time.time()
        torch.cuda.synchronize()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    if dist:
        dist.barrier()

    # timing of one launch kind on its own: back to back over rotating copies
    # inside a CUDA graph (chained with programmatic dependent launch, as in
    # the step), CUDA events around every replay, on the launching stream
    def time_graph(g, launches, replays):
        with torch.cuda.stream(stream):
            g.replay()
            stream.synchronize()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(replays)]
            for a_, b_ in evs:
                a_.record(stream)
                g.replay()
                b_.record(stream)
            stream.synchronize()
        return [a_.elapsed_time(b_) / launches for a_, b_ in evs]

    # enough distinct copies of every blob that one pass over a group streams
    # >= 512 MB (4x the L2), so no launch finds its weights in L2
    ncopy = {}
    for _, kind in GROUPS:
        gb = sum(len(layer[i]["blob"]) for i in group_members(layer, kind))
        ncopy[kind] = max(REPLICAS, -(-L2_ROTATION_BYTES // gb))
    ncopy_max = max(ncopy.values())
    copies = [reps[r] for r in range(REPLICAS)] + [[b.clone() for b in reps[0]] for _ in range(ncopy_max - REPLICAS)]

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    replays = max(5, min(50, args.steps // 400))
    per_group = {}
    for gname, kind in GROUPS:
        n = ncopy[kind]
        g = capture(lambda: [launch_group(lbq, layer, kind, copies[r], xs, ys, pdl=True) for r in range(n)])
        per_group[kind] = time_graph(g, n, replays)
        del g
    # per call: each matrix alone, chained over its own rotating copies
    per_call = []
    for i, e in enumerate(layer):
        n = max(REPLICAS, -(-L2_ROTATION_BYTES // len(e["blob"])))
        extra = [reps[0][i].clone() for _ in range(max(0, n - ncopy_max))]
        blobs = [copies[r % ncopy_max][i] for r in range(min(n, ncopy_max))] + extra
        g = capture(lambda: [launch(lbq, e, b, xs[i], ys[i], pdl=True) for b in blobs])
        per_call.append(time_graph(g, len(blobs), replays))
        del g, extra
    refinement = run_refinement(lbq, layer, dev, stream)
    kv_cache = time_kv_cache(lbq, dev, stream)
    decode_sweep = run_decode_sweep(lbq, layer, copies, ncopy, xs, ys, stream, replays)
    small_m = None if args.no_smallm_sweep else run_smallm_sweep(lbq, dev, stream)
    clk = clocks.summary(t_wall0, t_wall1, w_wall0, time.time())
    sweep70b = None
    if not args.no_sweep70b:
        sweep70b = run_sweep70b(lbq, dev, stream)
    clocks.stop()
    assert lbq.device_error(stream) == 0

    # e2e: host (pinned) activations in, outputs back to host, through the same
    # graph, one synchronisation per step (a decode step needs its result)
    h_x = torch.from_numpy(np.concatenate([np.ascontiguousarray(e["x"], dtype=np.float16).reshape(-1)
                                           for e in layer])).pin_memory()
    h_y = torch.empty(y_all.numel(), dtype=torch.float16).pin_memory()
    h2d = h_x.numel() * 2
    d2h = h_y.numel() * 2
    e2e_steps = max(10, min(2000, args.steps // 10))
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for s in range(e2e_steps):
            x_all.copy_(h_x, non_blocking=True)
            graphs[s % REPLICAS].replay()
            h_y.copy_(y_all, non_blocking=True)
            stream.synchronize()
        e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    e2e_value = whole_job_gbs(step_bytes, world, e2e_steps, e2e_s)

    peak, peak_kind = load_peaks()
    ms_step = ms_total / args.steps
    value = whole_job_gbs(step_bytes, world, args.steps, ms_total * 1e-3)
    groups_detail = []
    for gname, kind in GROUPS:
        gbytes = sum(layer[i]["bytes"] for i in group_members(layer, kind))
        us = statistics.mean(per_group[kind]) * 1e3
        groups_detail.append({"launch": gname, "matrices": [layer[i]["name"] for i in group_members(layer, kind)],
                              "bytes": gbytes, "us_per_launch": round(us, 3),
                              "GB_s": round(gbytes / (us * 1e-6) / 1e9, 1),
                              "frac_of_peak": round(gbytes / (us * 1e-6) / 1e9 / peak, 4)})
    dom = max(groups_detail, key=lambda d: d["us_per_launch"])
    achieved = dom["GB_s"]
    detail = []
    for i, e in enumerate(layer):
        us = statistics.median(per_call[i]) * 1e3
        gbs = e["bytes"] / (us * 1e-6) / 1e9
        detail.append({"kernel": e["kind"], "linear": e["name"], "N": e["N"], "K": e["K"], "n_out": e["n_out"],
                       "M": e["M"], "us_per_call": round(us, 3), "GB_s": round(gbs, 1),
                       "frac_of_peak": round(gbs / peak, 4)})
    w4_bytes = sum(e["bytes"] for e in layer if e["kind"] == "w4")
    w2_bytes = sum(e["bytes"] for e in layer if e["kind"] == "w2")
    us_w4 = statistics.mean(per_group["w4"]) * 1e3
    us_w2 = statistics.mean(per_group["w2"]) * 1e3
    capture_ok = kernel_source_hash() == TRAFFIC_CAPTURE["kernel_sha256_prefix"]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "dtype_detail": "4-/2-bit weights and fp16 activations in, exact fp16 products, fp32 accumulation",
        "data": "synthetic (seeded; shapes and distributions of the decode configs)",
        "config": config_dict(),
        "gpu_launches": launches_per_step * args.steps,
        "step_bytes": step_bytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": TRAFFIC_CAPTURE["traffic"].get(dom["launch"]) if capture_ok else None,
                     "kernel": "lbq_gemv_kernel, grouped launch %s (%d B algorithmic per launch): launches back to "
                               "back in a CUDA graph over rotating copies, CUDA events around each replay, "
                               "average per launch" % (dom["launch"], dom["bytes"]),
                     "peak_source": peak_kind},
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "detail": {"per_launch": groups_detail, "per_call": detail,
                   "implied_tokens_per_s": {
                       "llama3_8b_w4_32_layers_from_layer_sweep": round(1.0 / (32 * us_w4 * 1e-6), 1),
                       "llama3_8b_w2_32_layers_from_layer_sweep": round(1.0 / (32 * us_w2 * 1e-6), 1),
                       "llama3_8b_w4_32_layers_from_per_call": round(
                           1.0 / (32 * sum(statistics.median(per_call[i]) for i, e in enumerate(layer)
                                           if e["kind"] == "w4") * 1e-3), 1)},
                   "w4_layer_bytes": w4_bytes, "w2_layer_bytes": w2_bytes,
                   "decode_sweep_dependent_launches": decode_sweep, "small_m": small_m,
                   "llama3_70b_sweep": sweep70b, "selective_refinement": refinement, "kv_cache_4bit": kv_cache},
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


REFINE_K = 16   # channels per 1,024-channel chunk (1.6 % of the input channels)


def run_refinement(lbq, layer, dev, stream, replays=20):
    """Selective refinement after each 4-bit linear of the layer: select the
    REFINE_K largest |x_i| of every 1,024-channel chunk, then add their 4-bit
    residual columns (C = Q4(W - W_hat)).  Timed as select + apply, chained in
    a CUDA graph over rotating copies of the refinement blob (>= 512 MB), so the
    gathered columns come from HBM."""
    import torch
    out = {"k_per_chunk": REFINE_K, "per_linear": []}
    total_us = 0.0

    def timed(fn, copies):
        with torch.cuda.stream(stream):
            for c in copies[:2]:
                fn(c)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in copies:
                    fn(c)
            g.replay()
            stream.synchronize()
            ts = []
            for _ in range(replays):
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                g.replay()
                b_.record(stream)
                b_.synchronize()
                ts.append(a_.elapsed_time(b_) * 1e3 / len(copies))
        del g
        return statistics.median(ts)

    rblobs = []
    for e in layer:
        if e["kind"] != "w4":
            continue
        N, K = e["N"], e["K"]
        R = (synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W4, layer_id=e["li"]) - lbq.dequant_host(e["blob"]))
        rblob = lbq.pack_refine(R.astype(np.float32))
        rblobs.append(rblob)
        del R
        n_sel = lbq.refine_selected_count(K, REFINE_K)
        ncopy = max(2, min(64, -(-L2_ROTATION_BYTES // rblob.size)))
        d0 = torch.from_numpy(rblob).to(dev)
        copies = [d0] + [d0.clone() for _ in range(ncopy - 1)]
        x = torch.from_numpy(np.ascontiguousarray(e["x"]).reshape(-1)).to(dev)
        y = torch.zeros(N, dtype=torch.float32, device=dev)
        idx = torch.empty(n_sel, dtype=torch.int32, device=dev)

        def two_call(c):
            lbq.refine_select(x, K, REFINE_K, idx, stream=stream)
            lbq.refine_apply(c, N, K, x, idx, n_sel, y, stream=stream)

        us = timed(two_call, copies)
        cb = lbq.lib().lbq_refine_packed_bytes(N, 1) - 64
        nbytes = n_sel * cb + 2 * K + 6 * n_sel + 8 * N
        out["per_linear"].append({"linear": e["name"], "N": N, "K": K, "selected": n_sel,
                                  "us_per_call": round(us, 3), "bytes": nbytes,
                                  "GB_s": round(nbytes / (us * 1e-6) / 1e9, 1)})
        total_us += us
        del copies, d0
    assert lbq.device_error(stream) == 0
    torch.cuda.empty_cache()
    out["layer_us"] = round(total_us, 2)
    out["fused_layer"] = run_refined_sweep(lbq, [e for e in layer if e["kind"] == "w4"], rblobs, dev, stream, timed)
    return out


def run_refined_sweep(lbq, w4, rblobs, dev, stream, timed):
    """The 4-bit layer sweep with refinement fused: one grouped selection launch
    (the 7 activation vectors; chosen columns prefetched into L2) and one grouped
    GEMV launch that adds each row's correction (lbq_gemv_grouped_refined),
    against the plain grouped sweep, both over rotating copies of the weights and
    refinement blobs (>= 512 MB) in a CUDA graph."""
    import torch
    ncp = max(2, -(-L2_ROTATION_BYTES // sum(len(e["blob"]) + len(r) for e, r in zip(w4, rblobs))))
    blobs = [[torch.from_numpy(e["blob"]).to(dev) for e in w4] for _ in range(ncp)]
    rbs = [[torch.from_numpy(r).to(dev) for r in rblobs] for _ in range(ncp)]
    xs = [torch.from_numpy(np.ascontiguousarray(e["x"]).reshape(-1)).to(dev) for e in w4]
    ys = [torch.empty(e["N"], dtype=torch.float32, device=dev) for e in w4]
    nsel = [lbq.refine_selected_count(e["K"], REFINE_K) for e in w4]
    idxs = [torch.empty(n, dtype=torch.int32, device=dev) for n in nsel]

    def probs(c):
        return [(blobs[c][i], e["N"], e["K"], 0, xs[i], ys[i]) for i, e in enumerate(w4)]

    def plain(c):
        lbq.gemv_grouped(lbq.LBQ_KIND_W4, probs(c), pdl=True, stream=stream)

    def fused(c):
        lbq.refine_select_grouped([(xs[i], e["K"], REFINE_K, idxs[i], rbs[c][i], e["N"]) for i, e in enumerate(w4)],
                                  stream=stream)
        lbq.gemv_grouped_refined(lbq.LBQ_KIND_W4, probs(c), [(rbs[c][i], idxs[i], nsel[i]) for i in range(len(w4))],
                                 pdl=True, stream=stream)

    def select_only(c):
        lbq.refine_select_grouped([(xs[i], e["K"], REFINE_K, idxs[i], rbs[c][i], e["N"]) for i, e in enumerate(w4)],
                                  stream=stream)

    def gemv_only(c):
        lbq.gemv_grouped_refined(lbq.LBQ_KIND_W4, probs(c), [(rbs[c][i], idxs[i], nsel[i]) for i in range(len(w4))],
                                 pdl=True, stream=stream)

    us_plain = timed(plain, list(range(ncp)))
    us_fused = timed(fused, list(range(ncp)))
    us_sel = timed(select_only, list(range(ncp)))
    us_gemv = timed(gemv_only, list(range(ncp)))
    assert lbq.device_error(stream) == 0
    del blobs, rbs
    torch.cuda.empty_cache()
    return {"launches": 2, "us_plain_sweep": round(us_plain, 3), "us_refined_sweep": round(us_fused, 3),
            "retained_throughput": round(us_plain / us_fused, 4), "copies": ncp,
            "us_selection_alone": round(us_sel, 3), "us_refined_gemv_alone": round(us_gemv, 3)}


# a decode step can only group linears whose inputs are ready together:
# {q, k, v} (the layer input), o (after attention), {gate, up} (after o), down
# (after gate and up)
DECODE_STAGES = (("q_proj", "k_proj", "v_proj"), ("o_proj",), ("gate_proj", "up_proj"), ("down_proj",))


def run_decode_sweep(lbq, layer, copies, ncopy, xs, ys, stream, replays):
    """The layer sweep as a real decode step issues it: 4 grouped launches a layer
    (DECODE_STAGES), each depending on the one before (programmatic dependent
    launch: a launch's prologue overlaps the previous one, its activations are
    read after it completes), for the 4-bit and the 2-bit layer, over rotating
    copies of the weights in a CUDA graph."""
    import torch
    out = {}
    for kind in ("w4", "w2"):
        lk = lbq.LBQ_KIND_W2CB if kind == "w2" else lbq.LBQ_KIND_W4
        stages = [[i for i, e in enumerate(layer) if e["kind"] == kind and e["name"] in names] for names in DECODE_STAGES]
        n = ncopy[kind]

        def sweep():
            for r in range(n):
                for members in stages:
                    lbq.gemv_grouped(lk, group_args(lbq, layer, members, copies[r], xs, ys), M=1, pdl=True)
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                sweep()
            g.replay()
            stream.synchronize()
            ts = []
            for _ in range(replays):
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                g.replay()
                b_.record(stream)
                b_.synchronize()
                ts.append(a_.elapsed_time(b_) * 1e3 / n)
        del g
        us = statistics.median(ts)
        nbytes = sum(layer[i]["bytes"] for st in stages for i in st)
        out[kind] = {"launches_per_layer": len(stages), "us_per_layer": round(us, 3), "bytes": nbytes,
                     "GB_s": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "implied_tokens_per_s_32_layers": round(1.0 / (32 * us * 1e-6), 1)}
    assert lbq.device_error(stream) == 0
    return out


FMA_PEAK = 152 * 128 * 2.07e9       # FP32 FMA lanes of a GB300 (152 SMs x 128 a clock) at the 2.07 GHz maximum


def run_smallm_sweep(lbq, dev, stream, replays=5):
    """The batched 4-bit GEMM across M: the 4-bit gate (14336 x 4096) and down (4096 x 14336)
    projections at M = 2..64 (CUDA cores below 16, tensor cores from 16) and
    with their saliency-selected outlier columns at M = 16 / 64, the 2-bit ones
    with 3.5 % outlier columns (CUDA cores below 16, tensor cores from 16) and
    without outlier columns at M >= 16 (tensor cores).  Each
    configuration chained over
    rotating copies (>= 512 MB) in a CUDA graph.  Next to the HBM fraction: the
    FP32-FMA fraction below M = 16 (one FMA per weight and activation row) and
    the dense FP16 tensor fraction from M = 16."""
    import torch
    peaks = {}
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        with open(pp) as f:
            peaks = json.load(f)
    tc_peak = float(peaks.get("bf16_tflops", 1900.0)) * 1e12   # FP16 and BF16 dense rates are equal
    hbm_peak, _ = load_peaks()
    cases = []
    for li in (4, 6):
        name, N, K = synth.LLAMA3_8B_LINEARS[li]
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_SMALL_M, layer_id=li)
        b4 = lbq.pack_w4(W)
        for M in (2, 4, 8, 16, 32, 64):
            cases.append(("w4", name, N, K, M, 0, b4))
        idx4 = lbq.select_outliers_w4(W)                   # SPECTRA 3.2-3.3 saliency + kurtosis ratio
        b4o = lbq.pack_w4(W, idx4)
        for M in (16, 64):
            cases.append(("w4", name, N, K, M, len(idx4), b4o))
        W2 = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
        idx = lbq.select_outliers_impact(W2, synth.profile_vectors(K, workload=synth.WL_LLAMA8B_W2, layer_id=li), 0.035)
        b2o = lbq.pack_w2cb(W2, idx)
        for M in (2, 4, 8, 16, 32, 64):
            cases.append(("w2", name, N, K, M, len(idx), b2o))
        b2 = lbq.pack_w2cb(W2, np.zeros(0, np.int32))
        for M in (16, 64):
            cases.append(("w2", name, N, K, M, 0, b2))
        del W, W2
    rows = []
    for kind, name, N, K, M, n_out, blob in cases:
        n = max(REPLICAS, -(-L2_ROTATION_BYTES // blob.size))
        d0 = torch.from_numpy(blob).to(dev)
        cps = [d0] + [d0.clone() for _ in range(n - 1)]
        X = torch.from_numpy(synth.activations(M, K, workload=synth.WL_SMALL_M, layer_id=0)).to(dev)
        Y = torch.empty((M, N), dtype=torch.float16, device=dev)
        f = lbq.gemm_w4a16_smallM if kind == "w4" else lbq.gemm_w2cb_outlier_smallM
        with torch.cuda.stream(stream):
            for c in cps[:2]:
                f(c, M, N, K, n_out, X, K, Y, N, stream=stream, pdl=True)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in cps:
                    f(c, M, N, K, n_out, X, K, Y, N, stream=stream, pdl=True)
            g.replay()
            stream.synchronize()
            ts = []
            for _ in range(replays):
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                g.replay()
                b_.record(stream)
                b_.synchronize()
                ts.append(a_.elapsed_time(b_) * 1e3 / n)
        del g, cps, d0
        us = statistics.median(ts)
        nbytes = algorithmic_bytes(kind, N, K, n_out, M)
        gbs = nbytes / (us * 1e-6) / 1e9
        row = {"kind": kind, "linear": name, "N": N, "K": K, "M": M, "n_out": n_out,
               "path": "tensor cores" if M >= 16 else "CUDA cores",
               "us_per_call": round(us, 3), "GB_s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4)}
        macs = M * N * K
        if row["path"] == "CUDA cores":
            row["frac_of_fp32_fma"] = round(macs / (us * 1e-6) / FMA_PEAK, 4)
        else:
            row["frac_of_fp16_tensor"] = round(2 * macs / (us * 1e-6) / tc_peak, 4)
        rows.append(row)
    assert lbq.device_error(stream) == 0
    torch.cuda.empty_cache()
    return {"cases": rows, "fp32_fma_peak": FMA_PEAK, "fp16_tensor_peak_flops": tc_peak}


def run_sweep70b(lbq, dev, stream, replays=5):
    """The Llama-3-70B decode weight sweep: one decode token through every linear of a Llama-3-70B-shaped
    model (80 layers x 7 linears + lm_head, W4A16 G32, M = 1): 40.2 GB of packed
    weights streamed per token.  One layer is packed on the host (seeded, config
    5 distribution) and replicated 80 times in device memory, so every layer
    reads its own bytes; the lm_head is packed separately.  Timed as 81 grouped
    launches per token (one per layer, one for the lm_head) and as 561
    single-matrix launches, each captured in a CUDA graph with PDL chaining."""
    import torch
    t_pack = time.time()
    layer = []
    for li, (name, N, K) in enumerate(synth.LLAMA3_70B_LINEARS):
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA70B, layer_id=li)
        layer.append((name, N, K, torch.from_numpy(lbq.pack_w4(W)).to(dev)))
        del W
    hn, hN, hK = synth.LLAMA3_70B_LM_HEAD
    W = synth.weights_heavy_cols(hN, hK, workload=synth.WL_LLAMA70B, layer_id=99)
    head = torch.from_numpy(lbq.pack_w4(W)).to(dev)
    del W
    t_pack = time.time() - t_pack
    layers = [[b for (_, _, _, b) in layer]] + [[b.clone() for (_, _, _, b) in layer]
                                                for _ in range(synth.LLAMA3_70B_LAYERS - 1)]
    xs = {K: torch.from_numpy(synth.activations(1, K, workload=synth.WL_LLAMA70B, layer_id=K)[0]).to(dev)
          for K in sorted({K for (_, _, K, _) in layer} | {hK})}
    ys = [torch.empty(N, dtype=torch.float16, device=dev) for (_, N, _, _) in layer]
    yh = torch.empty(hN, dtype=torch.float16, device=dev)
    total = sum(algorithmic_bytes("w4", N, K, 0) for (_, N, K, _) in layer) * synth.LLAMA3_70B_LAYERS + \
        algorithmic_bytes("w4", hN, hK, 0)

    def token_grouped():
        for blobs in layers:
            lbq.gemv_grouped(lbq.LBQ_KIND_W4, [(blobs[i], N, K, 0, xs[K], ys[i])
                                               for i, (_, N, K, _) in enumerate(layer)], pdl=True)
        lbq.gemv_w4a16(head, hN, hK, 0, xs[hK], yh, pdl=True)

    def token_per_call():
        for blobs in layers:
            for i, (_, N, K, _) in enumerate(layer):
                lbq.gemv_w4a16(blobs[i], N, K, 0, xs[K], ys[i], pdl=True)
        lbq.gemv_w4a16(head, hN, hK, 0, xs[hK], yh, pdl=True)

    stages = [[i for i, (name, _, _, _) in enumerate(layer) if name in names] for names in DECODE_STAGES]

    def token_dependent():
        # what a decode step can group: {q, k, v} | o | {gate, up} | down, in order
        for blobs in layers:
            for members in stages:
                lbq.gemv_grouped(lbq.LBQ_KIND_W4, [(blobs[i], layer[i][1], layer[i][2], 0, xs[layer[i][2]], ys[i])
                                                   for i in members], pdl=True)
        lbq.gemv_w4a16(head, hN, hK, 0, xs[hK], yh, pdl=True)

    out = {"workload": "llama3_70b decode weight sweep: 80 x (q 8192x8192, k/v 1024x8192, o 8192x8192, gate/up "
                       "28672x8192, down 8192x28672) + lm_head 128256x8192, W4A16 G32, M=1, one token",
           "bytes_per_token": total, "host_pack_s": round(t_pack, 1),
           "note": "one packed layer replicated 80x in HBM (each layer streams its own copy)"}
    for label, fn, launches in (("fused_layer_sweeps", token_grouped, synth.LLAMA3_70B_LAYERS + 1),
                                ("dependent_launches", token_dependent, synth.LLAMA3_70B_LAYERS * 4 + 1),
                                ("per_call", token_per_call, synth.LLAMA3_70B_LAYERS * 7 + 1)):
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            g.replay()
            stream.synchronize()
            ts = []
            for _ in range(replays):
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                g.replay()
                b_.record(stream)
                b_.synchronize()
                ts.append(a_.elapsed_time(b_))
        ms = statistics.median(ts)
        out[label] = {"us_per_token": round(ms * 1e3, 1), "GB_s": round(total / (ms * 1e-3) / 1e9, 1),
                      "tokens_per_s": round(1e3 / ms, 1), "launches_per_token": launches}
        del g
    out["embedding_gather"] = time_embed_gather(lbq, head, hN, hK, dev, stream)
    assert lbq.device_error(stream) == 0
    del layers, head, layer
    torch.cuda.empty_cache()
    return out


KV_WIDTH = 1024            # Llama-3-8B: 8 KV heads x 128
KV_CONTEXT = 131072


def time_kv_cache(lbq, dev, stream, replays=10):
    """4-bit Group-32 KV cache of one Llama-3-8B layer tensor (width 1024): the
    quantise-on-write of one decode token (K and V: two calls), and the FP16
    read of a 131072-token cache (77.6 MB of records, 268 MB of FP16 rows)."""
    import torch
    rb = lbq.kv_record_bytes(KV_WIDTH)
    cache = torch.zeros((KV_CONTEXT, rb), dtype=torch.uint8, device=dev)
    rng = np.random.default_rng(7)
    states = torch.from_numpy(rng.standard_normal((KV_CONTEXT, KV_WIDTH)).astype(np.float16)).to(dev)
    lbq.kv_quantize(states, KV_CONTEXT, KV_WIDTH, cache, 0)               # fill the cache
    out = torch.empty((KV_CONTEXT, KV_WIDTH), dtype=torch.float16, device=dev)
    tok = [states[i:i + 1] for i in range(2)]

    def timed(fn, n):
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(n):
                    fn()
            g.replay()
            stream.synchronize()
            ts = []
            for _ in range(replays):
                a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a_.record(stream)
                g.replay()
                b_.record(stream)
                b_.synchronize()
                ts.append(a_.elapsed_time(b_) * 1e3 / n)
        return statistics.median(ts)

    us_w = timed(lambda: [lbq.kv_quantize(t, 1, KV_WIDTH, cache, KV_CONTEXT - 2 + i, stream=stream)
                          for i, t in enumerate(tok)], 50)
    us_r = timed(lambda: lbq.kv_dequant(cache, 0, KV_CONTEXT, KV_WIDTH, out, stream=stream), 5)
    read_bytes = KV_CONTEXT * (rb + 2 * KV_WIDTH)
    assert lbq.device_error(stream) == 0
    del cache, states, out
    torch.cuda.empty_cache()
    return {"width": KV_WIDTH, "record_bytes": rb,
            "append_one_token_k_and_v_us": round(us_w, 3),
            "read_context": KV_CONTEXT, "read_us": round(us_r, 2), "read_bytes": read_bytes,
            "read_GB_s": round(read_bytes / (us_r * 1e-6) / 1e9, 1)}


EMBED_TOKENS = 128


def time_embed_gather(lbq, table, V, D, dev, stream, batches=64, replays=10):
    """Fused embedding row gather (FP16 rows) of EMBED_TOKENS random token ids from
    a V x D 4-bit table; 64 different id batches per graph replay, so the rows
    come from HBM rather than L2."""
    import torch
    rng = np.random.default_rng(1234)
    ids = [torch.from_numpy(rng.integers(0, V, size=EMBED_TOKENS).astype(np.int32)).to(dev) for _ in range(batches)]
    out = torch.empty((EMBED_TOKENS, D), dtype=torch.float16, device=dev)
    with torch.cuda.stream(stream):
        lbq.embed_gather(lbq.LBQ_KIND_W4, table, V, D, 0, ids[0], out, stream=stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for b in ids:
                lbq.embed_gather(lbq.LBQ_KIND_W4, table, V, D, 0, b, out)
        g.replay()
        stream.synchronize()
        ts = []
        for _ in range(replays):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            g.replay()
            b_.record(stream)
            b_.synchronize()
            ts.append(a_.elapsed_time(b_) * 1e3 / batches)
    us = statistics.median(ts)
    nbytes = int(EMBED_TOKENS * D * (W4_BYTES_PER_WEIGHT + 2) + 4 * EMBED_TOKENS)
    return {"table": "%d x %d W4A16 G32 (the sweep's lm_head blob)" % (V, D), "tokens": EMBED_TOKENS,
            "us_per_call": round(us, 3), "bytes": nbytes, "GB_s": round(nbytes / (us * 1e-6) / 1e9, 1)}


def run_single(args):
    """One kernel configuration, launched steps times after warmup (for ncu captures)."""
    import torch
    from bit_weight_only_lbq_gb300 import lbq
    if args.single.startswith("sweep:"):
        return run_single_sweep(args, args.single.split(":")[1])
    if args.single.split(":")[0] in ("kv", "refine", "embed"):
        return run_single_row(args)
    kind, N, K, n_out, M = args.single.split(":")
    N, K, n_out, M = int(N), int(K), int(n_out), int(M)
    rng = np.random.default_rng(0)
    W = (rng.standard_normal((N, K), dtype=np.float32) * 0.02)
    idx = np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)
    blob = lbq.pack_w2cb(W, idx) if kind == "w2" else lbq.pack_w4(W, idx)
    del W
    e = dict(kind=kind, N=N, K=K, n_out=n_out, M=M)
    dev = torch.device("cuda", 0)
    d_blob = torch.from_numpy(blob).to(dev)
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float16)).to(dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    for _ in range(max(1, args.warmup)):
        launch(lbq, e, d_blob, x, y, pdl=False)
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch(lbq, e, d_blob, x, y, pdl=False)
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in ts]
    nbytes = algorithmic_bytes("w2" if kind == "w2" else "w4", N, K, n_out, M)
    assert lbq.device_error() == 0
    print(json.dumps({"single": args.single, "bytes": nbytes, "us_median": statistics.median(us),
                      "GB_s": nbytes / (statistics.median(us) * 1e-6) / 1e9}), flush=True)
    return 0


def run_single_row(args):
    """The KV cache read (kv:ROWS:WIDTH, after filling the cache), the refinement
    (refine:N:K:k, select + apply on a random residual) or the embedding row gather
    (embed:V:D:T, T random token ids of a random V x D 4-bit table, FP16 rows out),
    launched steps times after warmup without graphs (for ncu captures)."""
    import torch
    from bit_weight_only_lbq_gb300 import lbq
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(0)
    parts = args.single.split(":")
    if parts[0] == "kv":
        rows, width = int(parts[1]), int(parts[2])
        cache = torch.zeros((rows, lbq.kv_record_bytes(width)), dtype=torch.uint8, device=dev)
        states = torch.from_numpy(rng.standard_normal((rows, width)).astype(np.float16)).to(dev)
        lbq.kv_quantize(states, rows, width, cache, 0)
        out = torch.empty((rows, width), dtype=torch.float16, device=dev)
        fn = lambda: lbq.kv_dequant(cache, 0, rows, width, out)
        nbytes = rows * (lbq.kv_record_bytes(width) + 2 * width)
    elif parts[0] == "embed":
        V, D, T = int(parts[1]), int(parts[2]), int(parts[3])
        table = torch.from_numpy(lbq.pack_w4(rng.standard_normal((V, D), dtype=np.float32) * np.float32(0.02))).to(dev)
        ids = torch.from_numpy(rng.integers(0, V, size=T).astype(np.int32)).to(dev)
        out = torch.empty((T, D), dtype=torch.float16, device=dev)
        fn = lambda: lbq.embed_gather(lbq.LBQ_KIND_W4, table, V, D, 0, ids, out)
        nbytes = int(T * D * (W4_BYTES_PER_WEIGHT + 2) + 4 * T)
    else:
        N, K, k = int(parts[1]), int(parts[2]), int(parts[3])
        blob = torch.from_numpy(lbq.pack_refine((rng.standard_normal((N, K)) * 1e-3).astype(np.float32))).to(dev)
        x = torch.from_numpy(rng.standard_normal(K).astype(np.float16)).to(dev)
        y = torch.zeros(N, dtype=torch.float32, device=dev)
        n_sel = lbq.refine_selected_count(K, k)
        idx = torch.empty(n_sel, dtype=torch.int32, device=dev)

        def fn():
            lbq.refine_select(x, K, k, idx)
            lbq.refine_apply(blob, N, K, x, idx, n_sel, y)
        nbytes = n_sel * (lbq.lib().lbq_refine_packed_bytes(N, 1) - 64) + 2 * K + 6 * n_sel + 8 * N
    for _ in range(max(1, args.warmup)):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in ts]
    assert lbq.device_error() == 0
    print(json.dumps({"single": args.single, "bytes": nbytes, "us_median": statistics.median(us),
                      "GB_s": nbytes / (statistics.median(us) * 1e-6) / 1e9}), flush=True)
    return 0


def run_single_sweep(args, kind):
    """One grouped launch of the step (w4, w2 or w4m), launched steps times after
    warmup without graphs (for ncu captures of exactly that launch)."""
    import torch
    from bit_weight_only_lbq_gb300 import lbq
    layer = make_workload(lbq, 0)
    dev = torch.device("cuda", 0)
    blobs = [torch.from_numpy(e["blob"]).to(dev) if e["kind"] == kind else None for e in layer]
    xs = [torch.from_numpy(np.ascontiguousarray(e["x"])).to(dev) for e in layer]
    ys = [torch.empty((e["M"], e["N"]), dtype=torch.float16, device=dev) for e in layer]
    for _ in range(max(1, args.warmup)):
        launch_group(lbq, layer, kind, blobs, xs, ys, pdl=False)
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch_group(lbq, layer, kind, blobs, xs, ys, pdl=False)
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in ts]
    nbytes = sum(e["bytes"] for e in layer if e["kind"] == kind)
    assert lbq.device_error() == 0
    print(json.dumps({"single": args.single, "bytes": nbytes,
                      "launches": group_launch_count(lbq, layer, kind, blobs, xs, ys),
                      "us_median": statistics.median(us),
                      "GB_s": nbytes / (statistics.median(us) * 1e-6) / 1e9}), flush=True)
    return 0


def cpu_baseline() -> dict:
    """The oracle as it stands on the host cores, with inputs built by the oracle
    alone: (ii) dequantise-from-bytes + matvec over a row sample of every matrix of
    the step (the headline value, GB/s of algorithmic bytes), with (i) packing and
    (iii) matvec on the cached matrix beside it, and the Llama-3-70B sweep extrapolated."""
    rows = 128
    layer = oracle_workload(rows)
    step, _ = oracle_sample(layer, rows)
    t = time.perf_counter()
    step()
    dt = time.perf_counter() - t
    reps = max(1, min(20, int(10.0 / max(dt, 1e-3))))
    fig = oracle_figures(layer, rows, reps)
    return {"value": fig["dequant_matvec"]["GB_s"], "unit": "GB/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": "first %d rows of each of the step's 16 matrices, %d repetitions (FP64 NumPy; inputs and "
                      "outlier columns from the oracle)" % (rows, reps),
            "figures": fig, "llama3_70b_extrapolated": oracle_70b_extrapolated()}


if __name__ == "__main__":
    sys.exit(main())

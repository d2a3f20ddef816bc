#!/usr/bin/env python3
"""Throughput of the packed, padding-free (bi)LSTM forward + BPTT on GB300.

One step = pack (x and the upstream gradient) -> forward of every layer ->
BPTT of every layer -> unpack (y and dx), on one batch of synthetic
sequences already resident in HBM.  The metric counts non-padded frames:
N = sum of the sequence lengths per step (no padded frame is computed).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload k] [--impl ours|reference]

Prints one JSON line (rank 0).  With --gpus N > 1 (torchrun) every rank runs
an independent replica of the workload (weak scaling, no collective on the
data path); the time is the maximum over ranks.

Timing: CUDA events on the stream the library launches on, one pair per
step; L2 is flushed (a 512 MiB write) before every timed step, outside the
events.  SM clocks and throttle reasons are sampled with nvidia-smi during
the timed loop.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "non-padded frames/sec LSTM fwd+bwd (1 GB300); % of GEMM/SMEM roofline"
UNIT = "frames/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0, "source": "fallback"}
NUM_SMS = 152
FP32_LANES_PER_SM = 128


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    except Exception:
        return dict(FALLBACK_PEAKS)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"error": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"error": "no samples"}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for name, v in zip(names, r[4:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


# --------------------------------------------------------------------------- algorithmic work

def kind_work(kind: str, spec, rows: int, D0: int):
    """Algorithmic (flops, HBM bytes) of one step's launches of `kind`, summed over layers."""
    H, nd, e = spec.hidden_size, spec.num_directions, (2 if spec.dtype == "bf16" else 4)
    fl = by = 0.0
    for l in range(spec.num_layers):
        D = D0 if l == 0 else nd * H
        ex = e if l == 0 or spec.dtype == "bf16" else 4
        G4 = nd * 4 * H
        if kind == "input_gemm":
            fl += 2.0 * rows * D * G4
            by += rows * D * ex + G4 * D * e + rows * G4 * 4
        elif kind == "rec_fwd":
            fl += 8.0 * rows * H * H * nd
            by += 2 * rows * G4 * 4 + 2 * rows * nd * H * 4 + nd * 4 * H * H * e
        elif kind == "rec_bwd":
            fl += 8.0 * rows * H * H * nd
            by += 2 * rows * G4 * 4 + 3 * rows * nd * H * 4 + nd * 4 * H * H * e
        elif kind == "gemm_dx":
            fl += 2.0 * rows * G4 * D
            by += rows * G4 * 4 + G4 * D * e + rows * D * 4
        elif kind == "gemm_dw":
            fl += 2.0 * rows * G4 * D
            by += rows * G4 * 4 + rows * D * ex + G4 * D * 4
        elif kind == "gemm_dr":
            fl += 2.0 * rows * 4 * H * H * nd
            by += rows * G4 * 4 + rows * nd * H * 4 + nd * 4 * H * H * 4
        if kind == "convert":
            # bf16 operands of the tensor-core products (one K segment for bf16 layers, three for
            # fp32 layers): dA read once, written transposed and row-major; X, H_prev, W read and
            # written transposed; fp32 layers also split X and W for the input projection
            ns = 1 if spec.dtype == "bf16" else 3
            by += rows * G4 * 4 + rows * D * ex + rows * nd * H * 4 + G4 * D * e
            by += ns * 2 * (2 * rows * G4 + rows * D + rows * nd * H + G4 * D)
            if ns == 3:
                by += rows * D * 4 + G4 * D * 4 + ns * 2 * (rows * D + G4 * D)
    if kind == "pack":
        fl, by = 0.0, 2.0 * rows * (D0 * e + nd * H * 4)
    elif kind == "unpack":
        fl, by = 0.0, 2.0 * rows * (nd * H + D0) * 4
    return fl, by


SMEM_BYTES_PER_CLK = 128      # shared-memory bandwidth of one SM, bytes per clock
GEMM_KINDS = ("input_gemm", "gemm_dx", "gemm_dw", "gemm_dr")


def group_steps(lengths, slots):
    """Steps of each sequence group: the longest length among its sorted slots."""
    srt = np.sort(np.asarray(lengths))[::-1]
    slots = max(1, int(slots))
    return [int(srt[g]) for g in range(0, len(srt), slots)]


def rec_smem_bytes(kind, spec, rows, T, ctas, steps_per_cluster=None):
    """Algorithmic on-chip bytes of one recurrent pass over all layers.

    Per step of each cluster (one per direction and sequence group): every element of
    R_dir read once from on-chip storage (4H*H elements at the weight precision) plus the
    step's vector operand staged into each of the cluster's CTAs (its rows of H values:
    h_{t-1} forward, the partial sums of R^T*dA backward).  Summed over the clusters' steps:
    sum_g T_g * |R_dir| + ctas * N * H * b_h per direction (one group: T * |R_dir| + ...).
    """
    H, nd = spec.hidden_size, spec.num_directions
    e = 2 if spec.dtype == "bf16" else 4
    steps = float(sum(steps_per_cluster)) if steps_per_cluster else float(T)
    return float(spec.num_layers * nd * (steps * 4 * H * H * e + ctas * rows * H * e))


def roofline_of(kind, ms_per_step, calls_per_step, spec, rows, T, D0, peaks, rec_cfg, lengths=None):
    """Roofline entry of one kernel kind from its per-step time.

    rec_fwd/rec_bwd: shared-memory bandwidth of the SMs holding R (128 B/clk per SM at the
    maximum SM clock, over every CTA of every cluster in use: ctas x directions x groups).  GEMMs with bf16 operands (tcgen05):
    the sustained measured bf16 peak, or HBM when the bytes take longer.  The rest:
    HBM (measured copy bandwidth) or CUDA-core FP32 (derived) whichever bounds it.
    """
    fl, by = kind_work(kind, spec, rows, D0)
    sec = ms_per_step / 1e3
    clk = float(peaks.get("sm_max_mhz", 2070.0))
    per = max(1.0, calls_per_step)
    if kind in ("rec_fwd", "rec_bwd") and rec_cfg and rec_cfg.get("kernel") == "step_launches":
        # per-step tcgen05 products over the whole GPU (bf16 layers wider than one cluster)
        cpeak = float(peaks["bf16_tflops_sustained"])
        ach = fl / sec / 1e12 if sec > 0 else 0.0
        return {"kernel": kind, "bound": "tensor", "achieved": round(ach, 3), "peak": round(cpeak, 1),
                "unit": "TFLOP/s", "frac": round(ach / cpeak, 4), "recurrent_kernel": rec_cfg,
                "peak_source": "MEASURED_PEAKS.json sustained bf16",
                "per_launch": {"flops": fl / per, "ms": ms_per_step / per}}
    if kind in ("rec_fwd", "rec_bwd") and rec_cfg and rec_cfg.get("ctas_per_direction"):
        ctas = rec_cfg["ctas_per_direction"]
        groups = int(rec_cfg.get("groups") or 1)
        gsteps = group_steps(lengths, rec_cfg.get("slots_per_group") or len(lengths)) \
            if (lengths is not None and groups > 1) else None
        sb = rec_smem_bytes(kind, spec, rows, T, ctas, gsteps)
        sms = ctas * spec.num_directions * groups
        peak = sms * SMEM_BYTES_PER_CLK * clk * 1e6 / 1e9                     # GB/s
        ach = sb / sec / 1e9 if sec > 0 else 0.0
        tensor_peak = float(peaks["bf16_tflops_sustained"]) * (1.0 if spec.dtype == "bf16" else 1.1 / 2.25)
        out = {"kernel": kind, "bound": "smem", "achieved": round(ach, 1), "peak": round(peak, 1), "unit": "GB/s",
               "frac": round(ach / peak, 4), "recurrent_kernel": rec_cfg,
               "peak_source": f"derived: {sms} SMs x {SMEM_BYTES_PER_CLK} B/clk x {clk:.0f} MHz",
               "tensor_view": {"achieved_tflops": round(fl / sec / 1e12, 3) if sec > 0 else 0.0,
                               "peak_tflops": round(tensor_peak, 1)},
               "per_launch": {"smem_bytes": sb / per, "flops": fl / per, "ms": ms_per_step / per}}
        if gsteps:
            # the cluster of the longest sequences sets the kernel's time: its own bytes over its
            # own SMs (the other groups finish earlier and leave their SMs idle)
            H, nd = spec.hidden_size, spec.num_directions
            e = 2 if spec.dtype == "bf16" else 4
            srt = np.sort(np.asarray(lengths))[::-1]
            rows0 = int(srt[:int(rec_cfg["slots_per_group"])].sum())     # frames of group 0's slots
            b0 = float(spec.num_layers * (gsteps[0] * 4 * H * H * e + ctas * rows0 * H * e))
            p0 = ctas * SMEM_BYTES_PER_CLK * clk * 1e6 / 1e9
            a0 = b0 / sec / 1e9 if sec > 0 else 0.0
            out["critical_cluster"] = {"steps": gsteps[0], "rows": rows0, "achieved": round(a0, 1),
                                       "peak": round(p0, 1), "frac": round(a0 / p0, 4),
                                       "group_steps": gsteps}
        return out
    hbm_peak = float(peaks["hbm_gbs"])                                        # GB/s
    t_hbm = by / (hbm_peak * 1e9)
    if kind in GEMM_KINDS and spec.dtype == "bf16":
        cpeak, bound, src = float(peaks["bf16_tflops_sustained"]), "tensor", "MEASURED_PEAKS.json sustained bf16"
    elif kind in GEMM_KINDS and spec.input_size % 8 == 0:
        # fp32 products on tensor cores (three bf16 products): the fp32-input tensor rate, i.e. the
        # measured bf16 peak x the nominal tf32 / bf16 ratio (1.1 / 2.25 PFLOP/s)
        cpeak, bound = float(peaks["bf16_tflops_sustained"]) * 1.1 / 2.25, "tensor"
        src = "MEASURED_PEAKS.json sustained bf16 x 1.1/2.25 (nominal tf32/bf16)"
    elif kind == "convert":
        cpeak, bound, src = float("inf"), "hbm", ""
    else:
        cpeak, bound = NUM_SMS * FP32_LANES_PER_SM * 2 * clk * 1e6 / 1e12, "alu"
        src = "derived: 152 SMs x 128 FP32 lanes x 2 flop x max SM clock"
    t_c = fl / (cpeak * 1e12) if fl else 0.0
    if t_c >= t_hbm:
        ach = fl / sec / 1e12 if sec > 0 else 0.0
        return {"kernel": kind, "bound": bound, "achieved": round(ach, 3), "peak": round(cpeak, 1),
                "unit": "TFLOP/s", "frac": round(ach / cpeak, 4), "peak_source": src,
                "per_launch": {"flops": fl / per, "ms": ms_per_step / per}}
    ach = by / sec / 1e9 if sec > 0 else 0.0
    return {"kernel": kind, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(ach / hbm_peak, 4), "peak_source": f"MEASURED_PEAKS.json ({peaks.get('source')})",
            "per_launch": {"bytes": by / per, "ms": ms_per_step / per}}


# the sources that define each kernel kind's device code (a recorded ncu capture stays valid
# while these files are unchanged)
KERNEL_SOURCES = {
    "rec_fwd": ("recurrent_cluster.cu", "recurrent_cluster.cuh", "recurrent.cu", "recurrent.cuh", "tc_ptx.cuh",
                "common.cuh"),
    "rec_bwd": ("recurrent_cluster_bwd.cu", "recurrent_cluster.cuh", "recurrent.cu", "recurrent.cuh", "tc_ptx.cuh",
                "common.cuh"),
    "md_fwd": ("mdlstm.cu", "md_plan.cuh", "common.cuh"),
    "md_bwd": ("mdlstm.cu", "md_plan.cuh", "common.cuh"),
}


def code_only(text: str) -> str:
    """C/CUDA source without its comments and with whitespace runs collapsed: what the
    compiler sees, so that editing a comment does not retire a measurement."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                                   # string or character literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(kind: str = "") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "padding_free_variable_gb300", "csrc")
    files = KERNEL_SOURCES.get(kind) or tuple(sorted(os.listdir(csrc)))
    for f in sorted(files):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update((f + "\0" + code_only(fh.read()) + "\0").encode())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(f"{kind}@{workload}")
    if not ent or ent.get("source_digest") != source_digest(kind) or ent.get("workload") != workload:
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- CPU oracle arm

def oracle_sample(w, seconds: float, nthreads: int):
    """Sequences (caller order) forming a sample of about `seconds` of oracle work."""
    import oracle
    st = np.concatenate([[0], np.cumsum(w.lengths)])
    # calibrate on the shortest non-empty sequence
    cand = [int(i) for i in np.argsort(w.lengths, kind="stable") if w.lengths[i] > 0]
    i0 = cand[0]
    t0 = time.perf_counter()
    oracle.lstm_stack(w.lengths[[i0]], w.x[st[i0]:st[i0 + 1]], w.layers, w.spec.num_directions,
                      w.spec.hidden_size, G=w.G[st[i0]:st[i0 + 1]], nthreads=1)
    per_frame = (time.perf_counter() - t0) / max(1, int(w.lengths[i0]))
    budget_frames = seconds * nthreads / max(per_frame, 1e-9)
    seqs, frames = [], 0
    for i in range(len(w.lengths)):
        if w.lengths[i] == 0:
            continue
        if seqs and frames + w.lengths[i] > budget_frames:
            break
        seqs.append(i)
        frames += int(w.lengths[i])
    return seqs, frames


def run_oracle_on(w, seqs, nthreads):
    import oracle
    st = np.concatenate([[0], np.cumsum(w.lengths)])
    x = np.concatenate([w.x[st[s]:st[s + 1]] for s in seqs])
    G = np.concatenate([w.G[st[s]:st[s + 1]] for s in seqs])
    t0 = time.perf_counter()
    oracle.lstm_stack(w.lengths[seqs], x, w.layers, w.spec.num_directions, w.spec.hidden_size, G=G,
                      nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(w, seconds=15.0):
    import oracle
    oracle.build()
    nthreads = os.cpu_count() or 1
    seqs, frames = oracle_sample(w, seconds, nthreads)
    dt = run_oracle_on(w, seqs, nthreads)
    seqs1, frames1 = oracle_sample(w, seconds / 3, 1)
    dt1 = run_oracle_on(w, seqs1, 1)
    return {"value": round(frames / dt, 2), "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{len(seqs)} of {len(w.lengths)} sequences ({frames} frames), fwd+BPTT of every layer, "
                      f"fp64, OpenMP over sequences, {dt:.1f} s",
            "single_core": {"value": round(frames1 / dt1, 2), "unit": UNIT, "cores": 1,
                            "sample": f"{len(seqs1)} sequences ({frames1} frames), {dt1:.1f} s"}}


def reference_arm(args, w, config):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    nthreads = os.cpu_count() or 1
    per_step = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    seqs, frames = oracle_sample(w, per_step, nthreads)
    for _ in range(args.warmup):
        run_oracle_on(w, seqs, nthreads)
    times = [run_oracle_on(w, seqs, nthreads) for _ in range(args.steps)]
    total = sum(times)
    value = frames * args.steps / total
    out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": dict(config, sample_frames_per_step=frames),
           "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": nthreads, "kind": "oracle",
                            "sample": f"{len(seqs)} of {len(w.lengths)} sequences ({frames} frames) per step"},
           "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


# --------------------------------------------------------------------------- 2-D (MDLSTM) workloads

MD_METRIC = "non-padded pixels/sec MDLSTM layer fwd+bwd, 4 scan directions (1 GB300); % of CUDA-core roofline"
MD_UNIT = "pixels/s"


def md_kind_work(kind: str, N: int, nd: int, D: int, H: int) -> float:
    """Algorithmic flops of one call of an MDLSTM phase (every pixel, every direction).

    md_fwd: per cell the two recurrent products U1 h1 + U2 h2 (2 x 2 x 5H x H flops) and the
    cell (about 25 flops a unit); md_bwd: U1^T da + U2^T da of the successors (20 H^2) and the
    cell's backward (about 40 a unit); md_input: x W^T + b (2 N D 5H per direction);
    md_grads: dx and dW (2 N 5H D each per direction), dU1 and dU2 (2 N 5H H each per
    direction), db and the peephole sums (2 x 11H per cell)."""
    cells = N * nd
    if kind == "md_fwd":
        return cells * (20.0 * H * H + 25.0 * H)
    if kind == "md_bwd":
        return cells * (20.0 * H * H + 40.0 * H)
    if kind == "md_input":
        return 2.0 * N * D * nd * 5 * H
    if kind == "md_grads":
        return 2 * 2.0 * N * nd * 5 * H * D + 2 * 2.0 * cells * 5 * H * H + 22.0 * cells * H
    return 0.0


def md_cpu_sample(w, seconds: float, nthreads: int):
    """Images (in order) forming about `seconds` of oracle work, by pixel count."""
    import oracle
    oracle.build()
    probe = max(1, min(4, w.heights.size))
    pix_off = np.concatenate([[0], np.cumsum(w.heights.astype(np.int64) * w.widths)])
    t0 = time.perf_counter()
    run_md_oracle(w, list(range(probe)), pix_off)
    per_pixel = (time.perf_counter() - t0) / max(1, int(pix_off[probe]))
    budget = int(seconds / max(per_pixel, 1e-9))
    pick, tot = [], 0
    for i in range(w.heights.size):
        npx = int(pix_off[i + 1] - pix_off[i])
        if pick and tot + npx > budget:
            break
        pick.append(i)
        tot += npx
    return pick, tot, pix_off


def run_md_oracle(w, pick, pix_off):
    import oracle
    rows = np.concatenate([np.arange(pix_off[i], pix_off[i + 1]) for i in pick]) if pick else np.zeros(0, int)
    t0 = time.perf_counter()
    oracle.md_layer(w.heights[pick], w.widths[pick], w.x[rows], w.layer, w.G[rows])
    return time.perf_counter() - t0


def md_main(args):
    from padding_free_variable_gb300 import synthetic
    name = args.workload[3:]
    w = synthetic.md_workload(name, batch=args.batch or None)
    nd, D, H = w.num_directions, w.input_size, w.hidden_size
    N, B = w.N, int(w.heights.size)
    config = {"workload": w.name, "images": B, "pixels_per_step": N, "input_size": D, "hidden_size": H,
              "directions": nd, "dtype": "f32", "heights": f"uniform int [{w.heights.min()}, {w.heights.max()}]",
              "widths": f"uniform int [{w.widths.min()}, {w.widths.max()}]",
              "schedule": "diagonal (every image from step 0; the canvas schedule is a comparator)",
              "l2": "flushed (512 MiB write) before every timed step", "parallelism": "single GPU"}
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        nthreads = os.cpu_count() or 1
        per_step = max(0.5, 150.0 / max(1, args.steps + args.warmup))
        pick, px, pix_off = md_cpu_sample(w, per_step, nthreads)
        for _ in range(args.warmup):
            run_md_oracle(w, pick, pix_off)
        times = [run_md_oracle(w, pick, pix_off) for _ in range(args.steps)]
        value = px * args.steps / sum(times)
        out = {"metric": MD_METRIC, "value": round(value, 2), "unit": MD_UNIT, "n_gpus": args.gpus,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / args.steps, 3),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic", "impl": "reference", "config": dict(config, sample_pixels_per_step=px),
               "cpu_baseline": {"value": round(value, 2), "unit": MD_UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{len(pick)} of {B} images ({px} pixels) per step, single thread"},
               "e2e": {"value": round(value, 2), "unit": MD_UNIT, "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(out))
        return 0

    import torch
    torch.cuda.set_device(local_rank)
    from padding_free_variable_gb300 import build as native, ops
    native.build()
    plan = ops.MdPlan(w.heights, w.widths, 0, nd, 1)
    layer = ops.MdLayer(plan, w.layer, D, H)
    x_dev = torch.from_numpy(w.x).cuda()
    G_dev = torch.from_numpy(w.G).cuda()
    y_dev = torch.empty((N, nd * H), device="cuda")
    dx_dev = torch.empty((N, D), device="cuda")
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(lay=layer, xx=x_dev, gg=G_dev, yy=y_dev, dd=dx_dev):
        lay.forward(xx, yy)
        lay.backward(xx, gg, dd)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if plan.poll() != 0:
        raise RuntimeError("device status set during warm-up")
    sampler = ClockSampler(gpu_index(local_rank))
    sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    launches0 = plan.launch_count()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = plan.launch_count() - launches0
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(step_ms)
    if plan.poll() != 0:
        raise RuntimeError("device status set during the timed region")
    value = N * args.steps / (total_ms / 1e3)

    # per-phase times (a separate traced pass) and their rooflines
    peaks = load_peaks()
    clk = float(peaks.get("sm_max_mhz", 2070.0))
    alu_peak = NUM_SMS * FP32_LANES_PER_SM * 2 * clk * 1e6 / 1e12
    plan.enable_timing(True)
    traced = max(3, min(10, args.steps))
    for _ in range(traced):
        flush.fill_(0.0)
        step()
    tim = plan.read_timing()
    plan.enable_timing(False)
    kernels = {}
    for kind, (ms, calls) in tim.items():
        if not calls:
            continue
        per_ms = ms / calls
        fl = md_kind_work(kind, N, nd, D, H)
        ach = fl / (per_ms / 1e3) / 1e12
        kernels[kind] = {"kernel": kind, "bound": "alu", "achieved": round(ach, 3), "peak": round(alu_peak, 1),
                         "unit": "TFLOP/s", "frac": round(ach / alu_peak, 4),
                         "peak_source": f"derived: {NUM_SMS} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {clk:.0f} MHz",
                         "per_launch": {"flops": fl, "ms": round(per_ms, 4)}, "ms_per_step": round(ms / traced, 4)}
    dom = max(kernels.values(), key=lambda r: r["ms_per_step"])
    roof = {k: dom[k] for k in ("bound", "achieved", "peak", "unit", "frac", "kernel", "peak_source")}
    roof["traffic"] = recorded_traffic(dom["kernel"], w.name)
    walk = {"steps": plan.steps, "cells_per_step": round(N * nd / max(1, plan.steps), 1)}
    if "md_fwd" in kernels:
        walk["us_per_step_fwd"] = round(1e3 * kernels["md_fwd"]["per_launch"]["ms"] / max(1, plan.steps), 3)
    if "md_bwd" in kernels:
        walk["us_per_step_bwd"] = round(1e3 * kernels["md_bwd"]["per_launch"]["ms"] / max(1, plan.steps), 3)

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    x_host = torch.from_numpy(w.x).pin_memory()
    G_host = torch.from_numpy(w.G).pin_memory()
    y_host = torch.empty((N, nd * H), dtype=torch.float32).pin_memory()
    dx_host = torch.empty((N, D), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.fill_(float(i))
        es[i].record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        G_dev.copy_(G_host, non_blocking=True)
        step()
        y_host.copy_(y_dev, non_blocking=True)
        dx_host.copy_(dx_dev, non_blocking=True)
        ee[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in zip(es, ee))
    e2e = {"value": round(N * e2e_steps / (e2e_ms / 1e3), 2), "unit": MD_UNIT,
           "h2d_bytes_per_step": int(4 * (x_host.numel() + G_host.numel())),
           "d2h_bytes_per_step": int(4 * (y_host.numel() + dx_host.numel()))}

    comparators = {}
    if not args.no_comparators:
        csteps = max(3, min(10, args.steps))
        # the same cells on the page's canvas: a cell runs at its skewed canvas column
        cplan = ops.MdPlan(w.heights, w.widths, 0, nd, 0)
        clayer = ops.MdLayer(cplan, w.layer, D, H)
        cms = _time_steps(lambda: step(lay=clayer), csteps, flush, stream)
        comparators["canvas_schedule"] = {
            "pixels_per_s": round(N / (cms / 1e3), 2), "ms_per_step": round(cms, 3), "steps": cplan.steps,
            "canvas": {"height": cplan.canvas[0], "width": cplan.canvas[1], "rows": cplan.rows,
                       "fill": round(N / max(1, cplan.canvas[0] * cplan.canvas[1]), 4),
                       "skewed_fill": round(N / max(1, cplan.canvas[0] * (cplan.canvas[1] + cplan.canvas[0] - 1)),
                                            4)}}
        del clayer, cplan
        # the page's batch padding: every image padded to the batch's largest height and width
        # (the same kernels over B x hmax x wmax pixels; the work is what is compared)
        hm, wm = int(w.heights.max()), int(w.widths.max())
        Np = B * hm * wm
        pplan = ops.MdPlan(np.full(B, hm), np.full(B, wm), 0, nd, 0)
        player = ops.MdLayer(pplan, w.layer, D, H)
        xp = torch.zeros((Np, D), device="cuda")
        gp = torch.zeros((Np, nd * H), device="cuda")
        yp = torch.empty((Np, nd * H), device="cuda")
        dxp = torch.empty((Np, D), device="cuda")
        pms = _time_steps(lambda: step(lay=player, xx=xp, gg=gp, yy=yp, dd=dxp), csteps, flush, stream)
        comparators["batch_padded"] = {"pixels_per_s": round(N / (pms / 1e3), 2), "ms_per_step": round(pms, 3),
                                       "computed_pixels": Np, "waste_fraction": round((Np - N) / Np, 4),
                                       "zero_padding_rate": round((Np - N) / N, 4)}
        del player, pplan, xp, gp, yp, dxp

    cpu = None
    if not args.no_cpu_baseline:
        pick, px, pix_off = md_cpu_sample(w, 15.0, 1)
        dt = run_md_oracle(w, pick, pix_off)
        cpu = {"value": round(px / dt, 2), "unit": MD_UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{len(pick)} of {B} images ({px} pixels), fwd+backward of the layer in all "
                         f"{nd} directions, fp64, single thread, {dt:.1f} s"}

    out = {"metric": MD_METRIC, "value": round(value, 2), "unit": MD_UNIT, "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
           "clocks": clocks, "e2e": e2e, "gpu_launches": int(launches), "roofline": roof, "cpu_baseline": cpu,
           "kernels": kernels, "wavefront": walk, "comparators": comparators,
           "wall_s_timed_region": round(wall, 3),
           "step_ms": {"min": round(min(step_ms), 4), "median": round(statistics.median(step_ms), 4),
                       "max": round(max(step_ms), 4)}}
    print(json.dumps(out))
    return 0


# --------------------------------------------------------------------------- GPU arm

def _time_steps(fn, steps, flush, stream):
    import torch
    fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (a, b) in enumerate(ev):
        flush.fill_(float(i))
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def bucket_comparator(w, spec, bf16, layers, flush, stream, steps, width=100):
    """Sorted-bucket batching ("On batching variable size inputs", Sec. 2): sequences grouped
    by length into buckets of `width` frames, each bucket padded to its own longest sequence
    and run as its own batch (a padded plan) with the same kernels; one step = every bucket."""
    import torch
    from padding_free_variable_gb300 import ops
    from padding_free_variable_gb300.sharding import shard_rows
    lengths = np.asarray(w.lengths)
    lo = int(lengths.min()) // width * width
    groups = {}
    for i, L in enumerate(lengths):
        groups.setdefault((int(L) - lo) // width, []).append(i)
    xdt = torch.bfloat16 if bf16 else torch.float32
    runs, computed = [], 0
    for k in sorted(groups):
        idx = np.array(groups[k], dtype=np.int64)
        rows = shard_rows(lengths, idx)
        plan = ops.Plan(lengths[idx], padded=True)
        st = ops.PackedLSTMStack(plan, layers, spec.input_size, spec.hidden_size, spec.num_directions, bf16)
        x = torch.from_numpy(w.x[rows]).to("cuda", dtype=xdt)
        G = torch.from_numpy(w.G[rows]).cuda()
        runs.append((plan, st, x, G))
        computed += len(idx) * int(lengths[idx].max())

    def step():
        for plan, st, x, G in runs:
            st.step(x, G)

    ms = _time_steps(step, steps, flush, stream)
    N = int(lengths.sum())
    return {"frames_per_s": round(N / (ms / 1e3), 2), "ms_per_step": round(ms, 3), "bucket_width": width,
            "buckets": len(runs), "computed_frames": int(computed),
            "zero_padding_rate": round((computed - N) / N, 4), "waste_fraction": round((computed - N) / computed, 4)}


def stepwise_comparator(w, spec, bf16, layers, x_dev, G_dev, y_cat, dx_cat, flush, stream, steps):
    """The per-step-launch path (one product launch per direction and one cell launch per time
    step, the RETURNN paper's Sec. 4.2 design) on the same packed batch."""
    from padding_free_variable_gb300 import ops
    plan = ops.Plan(w.lengths)
    st = ops.PackedLSTMStack(plan, layers, spec.input_size, spec.hidden_size, spec.num_directions, bf16,
                             stepwise=True)

    def step():
        plan.pack(x_dev, st.x_packed)
        plan.pack(G_dev, st.dy_packed)
        st.forward_packed()
        st.backward_packed()
        plan.unpack(st.y[-1], y_cat)
        plan.unpack(st.dx[0], dx_cat)

    l0 = plan.launch_count()
    ms = _time_steps(step, steps, flush, stream)
    per_step = (plan.launch_count() - l0) // (steps + 1)
    return {"frames_per_s": round(w.N / (ms / 1e3), 2), "ms_per_step": round(ms, 3), "launches_per_step": per_step}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="3",
                    help="1..5: the 1-D LSTM workloads; md-words / md-lines: one 2-D MDLSTM layer over "
                         "example-packed images")
    ap.add_argument("--batch", type=int, default=0,
                    help="diagnostic: the workload with only this many sequences (same distributions); "
                         "0 = the workload as defined")
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-comparators", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cluster-variant", type=int, default=-1,
                    help="diagnostic: force the cluster recurrent kernels' variant (bit 0 bulk exchange, "
                         "bit 1 TMA tiles); -1 = the library's own choice")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if str(args.workload).startswith("md-"):
        return md_main(args)
    args.workload = int(args.workload)

    from padding_free_variable_gb300 import synthetic
    w = synthetic.workload(args.workload, batch=args.batch or None)
    spec = w.spec
    N, T, B = w.N, w.T, len(w.lengths)
    config = {"workload": spec.name, "sequences": B, "frames_per_step": N, "max_length": T,
              "input_size": spec.input_size, "hidden_size": spec.hidden_size, "layers": spec.num_layers,
              "directions": spec.num_directions, "gemm_operands": spec.dtype, "state": "f32",
              "lengths": str(spec.lengths), "seed": w.seed, "l2": "flushed (512 MiB write) before every timed step",
              "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}
    if args.cluster_variant >= 0:
        config["cluster_variant_forced"] = args.cluster_variant
    if args.impl == "reference":
        return reference_arm(args, w, config)

    import torch
    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from padding_free_variable_gb300 import build as native, ops
    if rank == 0:
        native.build()
    if dist:
        dist.barrier()

    bf16 = spec.dtype == "bf16"
    xdt = torch.bfloat16 if bf16 else torch.float32
    plan = ops.Plan(w.lengths)
    if args.cluster_variant >= 0:
        plan.debug_cluster_variant(args.cluster_variant)
    stack = ops.PackedLSTMStack(plan, ops.device_layers(w.layers, bf16), spec.input_size, spec.hidden_size,
                                spec.num_directions, bf16)
    x_dev = torch.from_numpy(w.x).to("cuda", dtype=xdt)
    G_dev = torch.from_numpy(w.G).cuda()
    y_cat = torch.empty((N, spec.num_directions * spec.hidden_size), device="cuda")
    dx_cat = torch.empty((N, spec.input_size), device="cuda")
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        plan.pack(x_dev, stack.x_packed)
        plan.pack(G_dev, stack.dy_packed)
        stack.forward_packed()
        stack.backward_packed()
        plan.unpack(stack.y[-1], y_cat)
        plan.unpack(stack.dx[0], dx_cat)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = plan.poll()
    if st != 0:
        raise RuntimeError(f"device status {st} during warm-up")

    # ---- timed region: K steps, per-step events, L2 flushed before each
    sampler = ClockSampler(gpu_index(local_rank))
    sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = plan.launch_count()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = plan.launch_count() - launches0
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    if plan.poll() != 0:
        raise RuntimeError("device status set during the timed region")
    from padding_free_variable_gb300.sharding import timing_over_ranks
    value, total_ms = timing_over_ranks(total_ms, N, args.steps, dist)

    # ---- per-kernel times (separate traced pass) for the roofline
    peaks = load_peaks()
    plan.enable_timing(True)
    traced = max(3, min(20, args.steps))
    for _ in range(traced):
        flush.fill_(0.0)
        step()
    tim = plan.read_timing()
    plan.enable_timing(False)
    kernels = {}
    rec_cfg = {"rec_fwd": plan.recurrent_config(False), "rec_bwd": plan.recurrent_config(True)}
    for k, bwd in (("rec_fwd", False), ("rec_bwd", True)):
        g, sl = plan.recurrent_groups(bwd)
        rec_cfg[k].update({"groups": g, "slots_per_group": sl})
    for kind, (ms, calls) in tim.items():
        if calls:
            r = roofline_of(kind, ms / traced, calls / traced, spec, plan.rows, T, spec.input_size, peaks,
                            rec_cfg.get(kind), lengths=w.lengths)
            r["ms_per_step"] = round(ms / traced, 4)
            kernels[kind] = r
    dom = max(kernels.values(), key=lambda r: r["ms_per_step"])
    roof = {k: dom[k] for k in ("bound", "achieved", "peak", "unit", "frac", "kernel", "peak_source")}
    roof["traffic"] = recorded_traffic(dom["kernel"], spec.name)
    recurrent = {}
    # per-step phases of the recurrent kernels from in-kernel clock64 stamps (CTA 0, direction 0)
    tsteps = min(T, 4096)
    tbuf = torch.zeros(2 * spec.num_directions * tsteps * 8, dtype=torch.int64, device="cuda")
    plan.trace_steps(tbuf, tsteps)
    step()
    torch.cuda.synchronize()
    plan.trace_steps(None, 0)
    stamps = tbuf.view(2, spec.num_directions, tsteps, 8).cpu().numpy().astype(np.float64)
    mhz = (clocks.get("sm_mhz") if isinstance(clocks, dict) else None) or float(peaks.get("sm_max_mhz", 2070.0))
    for kname, ki in (("fwd", 0), ("bwd", 1)):
        d = stamps[ki, 0]
        if not d[:, 0].any():
            continue
        us = lambda cyc: round(float(np.median(cyc)) / mhz, 3)
        # forward: 1 -> 2 stage h, 2 -> 5 product, 5 -> 3 cell; backward: 1 -> 2 cell (with the
        # peers' partial sums), 2 -> 5 partial product, 5 -> 3 gradient sums
        recurrent[f"phases_us_{kname}"] = {
            "barrier_wait": us(d[1:, 1] - d[1:, 0]), "after_barrier_to_2": us(d[:, 2] - d[:, 1]),
            "2_to_5": us(d[:, 5] - d[:, 2]), "5_to_3": us(d[:, 3] - d[:, 5]), "publish": us(d[:, 4] - d[:, 3]),
            "step": us(d[1:, 0] - d[:-1, 0]), "clock_mhz": mhz, "cta": 0, "direction": 0,
            "since_step_start": {str(k): us(d[:, k] - d[:, 0]) for k in range(1, 8) if d[:, k].any()}}
    if "rec_fwd" in kernels:
        recurrent["us_per_step_fwd"] = round(1e3 * kernels["rec_fwd"]["ms_per_step"] / (T * spec.num_layers), 3)
    if "rec_bwd" in kernels:
        recurrent["us_per_step_bwd"] = round(1e3 * kernels["rec_bwd"]["ms_per_step"] / (T * spec.num_layers), 3)

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    x_host = torch.from_numpy(w.x).to(xdt).pin_memory()
    G_host = torch.from_numpy(w.G).pin_memory()
    y_host = torch.empty(tuple(y_cat.shape), dtype=torch.float32).pin_memory()
    dx_host = torch.empty(tuple(dx_cat.shape), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 30))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush.fill_(float(i))
        es[i].record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        G_dev.copy_(G_host, non_blocking=True)
        step()
        y_host.copy_(y_cat, non_blocking=True)
        dx_host.copy_(dx_cat, non_blocking=True)
        ee[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(s.elapsed_time(e) for s, e in zip(es, ee))
    e2e = {"value": round(world * N * e2e_steps / (e2e_ms / 1e3), 2), "unit": UNIT,
           "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size() + G_host.numel() * 4),
           "d2h_bytes_per_step": int(y_host.numel() * 4 + dx_host.numel() * 4)}

    # ---- comparator: the same kernels on the zero-padded batch (masked)
    comparators = {}
    if not args.no_comparators and rank == 0:
        pplan = ops.Plan(w.lengths, padded=True)
        pstack = ops.PackedLSTMStack(pplan, stack.layers, spec.input_size, spec.hidden_size,
                                     spec.num_directions, bf16)
        psteps = max(3, min(10, args.steps))

        def pstep():
            pplan.pack(x_dev, pstack.x_packed)
            pplan.pack(G_dev, pstack.dy_packed)
            pstack.forward_packed()
            pstack.backward_packed()
            pplan.unpack(pstack.y[-1], y_cat)
            pplan.unpack(pstack.dx[0], dx_cat)
        pstep()
        torch.cuda.synchronize()
        ps = [torch.cuda.Event(enable_timing=True) for _ in range(psteps)]
        pe = [torch.cuda.Event(enable_timing=True) for _ in range(psteps)]
        for i in range(psteps):
            flush.fill_(float(i))
            ps[i].record(stream)
            pstep()
            pe[i].record(stream)
        torch.cuda.synchronize()
        pms = sum(s.elapsed_time(e) for s, e in zip(ps, pe)) / psteps
        comparators["zero_padded"] = {"frames_per_s": round(N / (pms / 1e3), 2), "ms_per_step": round(pms, 3),
                                      "computed_frames": int(B * T),
                                      "waste_fraction": round((B * T - N) / (B * T), 4),
                                      "zero_padding_rate": round((B * T - N) / N, 4)}
        del pstack, pplan
        comparators["sorted_buckets"] = bucket_comparator(w, spec, bf16, stack.layers, flush, stream, psteps)
        comparators["per_step_launch"] = stepwise_comparator(w, spec, bf16, stack.layers, x_dev, G_dev, y_cat,
                                                             dx_cat, flush, stream, max(3, min(5, args.steps)))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "bf16-operands/f32" if bf16 else "f32",
               "data": "synthetic", "config": config, "clocks": clocks, "e2e": e2e, "gpu_launches": int(launches),
               "roofline": roof, "cpu_baseline": cpu, "kernels": kernels, "recurrent": recurrent,
               "comparators": comparators, "wall_s_timed_region": round(wall, 3),
               "step_ms": {"min": round(min(step_ms), 4), "median": round(statistics.median(step_ms), 4),
                           "max": round(max(step_ms), 4)}}
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

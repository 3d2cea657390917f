#!/usr/bin/env python
"""Throughput of the routed-attention DiT denoising forward on GB300.

One step = one fresh denoiser step through the C ABI (h3dit_denoise_step):
bf16(z) -> all DiT blocks of the workload -> v = x_L -> z += dt v.  The
default workload is 50 blocks at 15,435 packed rows (512 text, 1,024 audio,
13,899 video; hidden 5,120, 40 heads x 128, MLP 4x GELU, top-k 16 of 218
video tiles + pooled branch), dt = -1/8.

Prints one JSON line (rank 0).  ``value`` = packed rows/s per DiT block over
the whole job (rows x blocks x steps x ranks / max-over-ranks time).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload forward50_15435_d5120|block_15435_d5120|block_4096_d3072|
                              loop20_4096_d3072|block_15435_d5376_swiglu|
                              forward50_15435_d5376_swiglu|block_15435_cubes_d5376_swiglu|
                              forward50_15435_cubes_d5376_swiglu|
                              sample50_15435_cubes_d5376_swiglu]

The sample50 workload runs one fresh pass of h3dit_sample_step instead: fp32 patch
projections of the video (96 channels) and audio (32) latents, the 50 blocks, the
final AdaLN and output heads with the Euler update fused.

The loop workload (20 Euler steps, 45 of 50 blocks, reuse 2) also prints a
top-k density sweep {4, 8, 16, 32, all 56 tiles} of one block.

--workload routed_attention_1024 (or attn_tiny_1024) times h3dit_routed_attention
alone on the 1,024-row, 4 x 64 case at top-k 4 and at top-k 16 (every tile: dense
attention), beside the CPU oracle on the same inputs.

The CPU baseline and --impl reference time the float32 C oracle (oracle/h3time.c,
plain loops, OpenMP on all host cores): the whole block when it fits the time
budget, else a uniform 1/s sample of it (every s-th 64-row chunk of rows through the
row-local stages, every s-th query tile and prefix chunk through attention, the
router over all tiles), reported as the rows processed per second.  Multi-GPU runs
are independent replicas (one per rank, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402

METRIC = ("packed rows/s per DiT block and s per 50-block forward, % of bf16 TC peak")
UNIT = "packed rows/s per block"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
KERNEL_SOURCES = {"gemm": ["gemm.cu", "ptx.cuh"], "attention": ["attention.cu", "ptx.cuh"]}


# ----------------------------------------------------------------------------- helpers
def workload(name):
    wl = S.workload_by_name(name)
    n_blocks = wl.n_blocks if wl.extra.get("forward") else 1
    return wl, n_blocks


def fc1_width(s):
    """Rows of the fc1 weight: 2F for the SwiGLU MLP (gate and up), F for GELU."""
    return 2 * s.mlp_width if s.mlp == "swiglu" else s.mlp_width


def block_weight_bytes(s):
    D, A, F = s.hidden, s.attn_width, s.mlp_width
    return 2 * (D * 4 * A + A * D + D * fc1_width(s) + F * D)


def block_flops(s):
    """Algorithmic flops of one block (2 per MAC): the four projections plus
    the attention the method performs (prefix rows over all N keys, video rows
    over the prefix and k selected tiles of V / Tv rows on average: 64-row slices,
    or clipped 4x4x4 cubes)."""
    N, D, A, F = s.n_rows, s.hidden, s.attn_width, s.mlp_width
    gemm = 2.0 * N * (D * 4 * A + A * D + D * fc1_width(s) + F * D)
    tv = s.n_video_tiles
    k = min(s.topk, tv)
    attn = 4.0 * s.head_dim * s.heads * (s.n_prefix * N + s.n_video * (s.n_prefix
                                                                       + k * s.n_video / tv))
    return gemm, attn


def reduced_shape(s):
    """The token-reduced section's shape: video grid T x H x ceil(W/2)."""
    T, Hg, Wg = s.video_grid
    Wr = (Wg + 1) // 2
    return s.with_(n_video=T * Hg * Wr, video_grid=(T, Hg, Wr), pair_w=Wg, token_reduction=False)


def block_shapes(s, n_blocks, reduction):
    """The shape of every block position of one step."""
    if not reduction or not (0 <= reduction[0] < reduction[1]) or reduction[0] >= n_blocks:
        return [s] * n_blocks
    rs = reduced_shape(s)
    return [rs if reduction[0] <= b < reduction[1] else s for b in range(n_blocks)]


def stage_flops(s):
    N, D, A, F = s.n_rows, s.hidden, s.attn_width, s.mlp_width
    _, attn = block_flops(s)
    return {"qkvg": 2.0 * N * D * 4 * A, "out_proj": 2.0 * N * A * D,
            "fc1": 2.0 * N * D * fc1_width(s), "fc2": 2.0 * N * F * D, "attention": attn}


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def source_sha(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "audio_diffusion_transformer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, stage, workload_name):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source
    is unchanged since it was captured; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            for ln in f:
                if ln.startswith("#") or not ln.strip():
                    continue
                k, st, wl, sha, nbytes = ln.split()[:5]
                if k == kernel and st == stage and wl == workload_name and sha == source_sha(kernel):
                    return int(float(nbytes))
    except (OSError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 10:
                    continue
                if self.bus_id and self.bus_id[-12:] not in parts[1].lower():
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = sorted(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": float(rows[0][3]) if rows[0][3].replace(".", "").isdigit() else None,
                "samples": len(rows), "reasons": reasons}


# ----------------------------------------------------------------------------- CPU oracle
def forward_config(wl, n_blocks, world):
    """The ``config`` object of a forward or sampler-step line (both arms print it)."""
    shape = wl.shape
    N, D = shape.n_rows, shape.hidden
    dt = -0.125
    shapes = block_shapes(shape, n_blocks, wl.extra.get("reduction"))
    return {"workload": wl.name, "n_rows": N, "n_text": shape.n_text,
            "n_audio": shape.n_audio, "n_video": shape.n_video, "n_blocks": n_blocks,
            "hidden": D, "heads": shape.heads, "head_dim": shape.head_dim,
            "attn_width": shape.attn_width,
            "mlp": (f"SwiGLU {shape.mlp_width}" if shape.mlp == "swiglu"
                    else f"{shape.mlp_width // D}x GELU"),
            "params_b": n_blocks * (D * 4 * shape.attn_width + shape.attn_width * D
                                    + D * fc1_width(shape) + shape.mlp_width * D) / 1e9,
            "topk": shape.topk, "tile": shape.tile,
            "video_tiles": (f"{shape.n_video_tiles} cubes "
                            f"{'x'.join(map(str, shape.cube))} of a "
                            f"{'x'.join(map(str, shape.video_grid))} grid, 3-D rotary"
                            if shape.video_grid else
                            f"{shape.n_video_tiles} slices of 64 rows"),
            "dt": dt, "parallelism": f"replicas x{world}",
            "rows_per_block": ({"full": N, "reduced": min(sb.n_rows for sb in shapes),
                                "reduced_blocks": list(wl.extra["reduction"])}
                               if len(set(sb.n_rows for sb in shapes)) > 1 else N),
            "step": ("sampler step on the modality latents: fp32 patch projections, "
                     "blocks, final AdaLN + output heads with the Euler update"
                     + (f", token reduction over blocks [{wl.extra['reduction'][0]}, "
                        f"{wl.extra['reduction'][1]})" if wl.extra.get("reduction")
                        else "")
                     if wl.extra.get("ends") else
                     "denoiser step on hidden-width latents: bf16(z), blocks, "
                     "z += dt x_L"),
            "l2": f"inputs larger than L2 (each block reads its own "
                  f"{block_weight_bytes(shape) / 1e6:.0f} MB of weights)"}


def _bf16_values(a):
    """float32 array rounded to the nearest bf16 value (ties to even), as float32."""
    import numpy as np
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def slice_shape(shape):
    """The float32 baseline tiles video rows as 64-row slices: a cube layout is timed
    at the same sizes with slice tiles (the same work up to the clipped cubes' fill)."""
    if getattr(shape, "video_grid", None):
        return shape.with_(video_grid=None, token_reduction=False)
    return shape


def cpu_block(shape, seed=0):
    """The float32 C block with seeded inputs of the workload's distributions: weights
    and biases bf16 N(0, 0.02) (input-major), modulation N(0, 0.1^2), q/k norm weights
    1 + N(0, 0.02), x bf16 N(0, 1)."""
    import numpy as np

    from oracle import ctime
    s = slice_shape(shape)
    rng = np.random.default_rng(seed)
    D, A, F, d = s.hidden, s.attn_width, s.mlp_width, s.head_dim
    F1 = fc1_width(s)

    def rn(*sz, std=0.02, mean=0.0, round_bf16=True):
        a = rng.standard_normal(sz, dtype=np.float32) * np.float32(std) + np.float32(mean)
        return _bf16_values(a) if round_bf16 else a

    w = {"w_qkvg": rn(D, 4 * A), "b_qkvg": rn(4 * A), "w_o": rn(A, D), "b_o": rn(D),
         "w1": rn(D, F1), "b1": rn(F1), "w2": rn(F, D), "b2": rn(D),
         "mod": rn(6, D, std=0.1, round_bf16=False), "qnorm_w": rn(d, mean=1.0),
         "knorm_w": rn(d, mean=1.0)}
    if getattr(s, "prefix_mod", False):
        w["mod_prefix"] = rn(6, D, std=0.1, round_bf16=False)
    blk = ctime.Block(s, w)
    blk.scratch.fill(0.0)  # touch every page before anything is timed
    x = rn(s.n_rows, D, std=1.0)
    return blk, x, s


def sampled_rows(n_rows, sample):
    """Rows that a 1/sample call runs through the row-local stages (every sample-th
    64-row chunk)."""
    return sum(min(64, n_rows - c * 64) for c in range(0, -(-n_rows // 64), sample))


def time_cpu_block(blk, x, sample):
    t0 = time.perf_counter()
    blk.run(x, sample=sample)
    return time.perf_counter() - t0


def cpu_sample_plan(blk, x, n_rows, budget_s):
    """Times a 1/16 calibration call and picks the smallest sample divisor s whose call
    should take about budget_s (1 = the whole block)."""
    t16 = time_cpu_block(blk, x, 16)
    est_full = t16 * n_rows / max(sampled_rows(n_rows, 16), 1)
    return max(1, math.ceil(est_full / budget_s)), est_full


def sample_desc(s, sample, n_rows):
    what = ("the whole block" if sample == 1 else
            f"a 1/{sample} sample of the block: rows of every {sample}th 64-row chunk "
            f"({sampled_rows(n_rows, sample)} of {n_rows}) through the norms, projections "
            f"and MLP, every {sample}th video query tile and prefix chunk through attention, "
            f"the router over all tiles")
    return (f"float32 C oracle (plain loops, OpenMP) on {s.n_rows} rows, hidden {s.hidden}, "
            f"{s.heads} x {s.head_dim}, top-k {s.topk}: {what}; value = rows processed / s")


def cpu_baseline(shape, budget_s=30.0):
    """Measured CPU baseline: the float32 C oracle on the whole block when that fits the
    budget, else on the smallest uniform sample that does."""
    from oracle import ctime
    blk, x, s = cpu_block(shape)
    sample, est = cpu_sample_plan(blk, x, s.n_rows, budget_s)
    if sample > 1 and est <= 1.5 * budget_s:
        sample = 1
    t = time_cpu_block(blk, x, sample)
    rows = sampled_rows(s.n_rows, sample)
    measured = "measured full block" if sample == 1 else f"measured 1/{sample} sample"
    return {"value": rows / t, "unit": UNIT, "cores": ctime.threads(),
            "kind": f"oracle fp32, {measured}", "sample": sample_desc(s, sample, s.n_rows),
            "s_per_block": t * s.n_rows / rows, "seconds_timed": t}


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value across the replicas (the job's wall time is the slowest rank's)."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's rows over the slowest rank's time."""
    return rows_per_rank * world / (max_ms / 1e3)


# ----------------------------------------------------------------------------- GPU arm
def make_blocks(torch, shape, n_blocks, seed, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    D, A, F, d = shape.hidden, shape.attn_width, shape.mlp_width, shape.head_dim
    blocks = []

    def rn(*sz, std=0.02, mean=0.0, dtype=torch.bfloat16):
        t = torch.randn(*sz, generator=g, device=dev, dtype=torch.float32)
        return (t * std + mean).to(dtype).contiguous()

    for _ in range(n_blocks):
        F1 = fc1_width(shape)
        blocks.append({"w_qkvg": rn(4 * A, D), "b_qkvg": rn(4 * A), "w_o": rn(D, A), "b_o": rn(D),
                       "w1": rn(F1, D), "b1": rn(F1), "w2": rn(D, F), "b2": rn(D),
                       "mod": rn(6, D, std=0.1, dtype=torch.float32),
                       "qnorm_w": rn(d, mean=1.0), "knorm_w": rn(d, mean=1.0)})
        if getattr(shape, "prefix_mod", False):
            blocks[-1]["mod_prefix"] = rn(6, D, std=0.1, dtype=torch.float32)
    return blocks


def make_ends(torch, shape, cv, ca, seed, dev):
    """Both ends on the device, same distributions as synthetic.ends_weights."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    D = shape.hidden

    def rn(*sz, std=1.0, dtype=torch.float32):
        return (torch.randn(*sz, generator=g, device=dev, dtype=torch.float32) * std).to(
            dtype).contiguous()

    e = {"c_video": cv, "c_audio": ca, "text": rn(max(shape.n_text, 1), D, dtype=torch.bfloat16)}
    for m, c in (("video", cv), ("audio", ca)):
        e[f"w_in_{m}"] = rn(c, D, std=0.1)
        e[f"b_in_{m}"] = rn(D, std=0.02)
        e[f"w_out_{m}"] = rn(c, D, std=0.02, dtype=torch.bfloat16)
        e[f"b_out_{m}"] = rn(c, std=0.02, dtype=torch.bfloat16)
        e[f"mod_out_{m}"] = rn(2, D, std=0.1)
    return e


FLOP_PER_CLK_SM = 8192  # dense bf16 tcgen05: one M=128 N=256 K=16 MMA per 128 cycles per SM


def per_clock_peak(n_sms, sm_mhz):
    """Dense bf16 tensor peak at the sampled SM clock, TFLOP/s (None without a clock)."""
    if not n_sms or not sm_mhz:
        return None
    return FLOP_PER_CLK_SM * n_sms * sm_mhz * 1e6 / 1e12


def dominant_kernel(shape, shapes, stages, K, workload_name, clk_peak=None, calls=None):
    """Roofline of the kernel with the largest stage time, from the live stage records
    (ms, kernel launches); achieved = its algorithmic flops / its time.  Also per-kernel
    rates.  ``calls``: how many times each block stage ran in the records (default: one
    per block position per step; a projection whose last round of tiles is split runs
    two kernels per call, its GEMM and the reduction of the split tiles, both timed in
    the stage).  ``clk_peak``: the tensor peak at the sampled SM clock
    (frac_per_clock)."""
    if calls is None:
        calls = len(shapes) * K
    pk, pk_kind = peaks()
    peak_tc = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    # per-launch flops of each stage, averaged over the block positions
    sf = {k: sum(stage_flops(sb)[k] for sb in shapes) / len(shapes)
          for k in stage_flops(shape)}
    fc1_name = "gemm<swiglu>" if shape.mlp == "swiglu" else "gemm<gelu>"
    groups = {"gemm<qkvg>": ["qkvg"], fc1_name: ["fc1"], "gemm<resid>": ["out_proj", "fc2"],
              "attention": ["attention"]}
    g_ms = {g: sum(stages[s_][0] for s_ in st) for g, st in groups.items()}
    dom = max(g_ms, key=g_ms.get)
    n_launch = calls * len(groups[dom])
    n_kernels = sum(stages[s_][1] for s_ in groups[dom])
    flops = sum(sf[s_] * calls for s_ in groups[dom])
    kernel = "attention" if dom == "attention" else "gemm"
    roofline = {"bound": "tensor", "kernel": dom,
                "achieved": flops / (g_ms[dom] / 1e3) / 1e12, "peak": peak_tc,
                "peak_kind": f"bf16 sustained, {pk_kind}", "unit": "TFLOP/s",
                "traffic": recorded_traffic(kernel, dom, workload_name),
                "launch_ms": g_ms[dom] / max(n_launch, 1), "launches": n_launch,
                "kernel_launches": n_kernels}
    roofline["frac"] = roofline["achieved"] / peak_tc
    if clk_peak:
        roofline["peak_per_clock"] = clk_peak
        roofline["frac_per_clock"] = roofline["achieved"] / clk_peak
    kernels = {}
    for g, st in groups.items():
        fl = sum(sf[s_] * calls for s_ in st)
        tf = fl / (g_ms[g] / 1e3) / 1e12 if g_ms[g] > 0 else None
        kernels[g] = {"ms_per_step": g_ms[g] / K, "tflops": tf,
                      "frac": tf / peak_tc if tf else None}
        if clk_peak and tf:
            kernels[g]["frac_per_clock"] = tf / clk_peak
    return roofline, kernels


def near_tie_audit(scores, idx, k, rel_gap=1e-5):
    """Near-ties of the router's top-k on the GPU's own fp32 tile scores [H, Tv, Tv]:
    (head, query tile) pairs whose k-th and (k+1)-th largest scores differ by less than
    rel_gap of the k-th (the pairs where two correct implementations may select
    differently).  Also checks that every selection [H, Tv, k] is a top-k of its scores
    under the (score desc, tile asc) order with NaN as -inf."""
    import numpy as np
    sc = np.where(np.isnan(scores), -np.inf, scores.astype(np.float64))
    H, T, n_keys = sc.shape
    order = np.argsort(-sc, axis=-1, kind="stable")  # ties: lower tile first
    srt = np.take_along_axis(sc, order, axis=-1)
    if k < n_keys:
        kth, nxt = srt[..., k - 1], srt[..., k]
        with np.errstate(invalid="ignore"):
            gap = (kth - nxt) / np.maximum(np.abs(kth), 1e-30)
        near = int(np.sum(gap < rel_gap))
    else:
        near = 0
    want = np.sort(order[..., :k], axis=-1)
    consistent = bool(np.array_equal(want, np.sort(idx, axis=-1)))
    return {"pairs": int(H * T), "near_ties": near, "rel_gap": rel_gap,
            "selections_are_topk_of_scores": consistent}


def block_near_ties(h3, torch, shape, weights, x_rows, dev):
    """Near-tie audit of one block at the bench's input: the block runs once with its
    intermediates kept, and its own tile scores and selections are read back."""
    cs = h3.make_shape(shape)
    cs = h3.make_shape(shape, cs.flags | h3.H3DIT_KEEP_INTERMEDIATES)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device=dev)
    x = x_rows.clone()
    h3.block_forward(cs, weights, x, ws)
    torch.cuda.synchronize()
    lay = h3.workspace_layout(cs)
    H, tv = shape.heads, shape.n_video_tiles
    k = min(shape.topk, tv)
    sc = ws[lay["scores"]:lay["scores"] + H * tv * tv * 4].view(torch.float32)
    ix = ws[lay["idx"]:lay["idx"] + H * tv * k * 4].view(torch.int32)
    out = near_tie_audit(sc.view(H, tv, tv).cpu().numpy(), ix.view(H, tv, k).cpu().numpy(), k)
    out["where"] = "block 0 at the bench input (the GPU's fp32 tile scores)"
    del ws
    return out


def timed_steps(torch, stream, step, K):
    """K steps with a CUDA event between consecutive steps on the launching stream:
    (total ms, per-step ms list)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    ev[0].record(stream)
    for i in range(K):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    return ev[0].elapsed_time(ev[K]), per


def median(xs):
    xs = sorted(xs)
    n = len(xs)
    return xs[n // 2] if n % 2 else 0.5 * (xs[n // 2 - 1] + xs[n // 2])


def run_ours(args, rank, world, local_rank):
    import torch

    import audio_diffusion_transformer_gb300 as h3
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl, n_blocks = workload(args.workload)
    shape = wl.shape
    N, D = shape.n_rows, shape.hidden
    cs = h3.make_shape(shape)
    ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device=dev)
    blocks = make_blocks(torch, shape, n_blocks, wl.seed + 1000 * rank, dev)
    ids = list(range(n_blocks))
    gz = torch.Generator(device=dev)
    gz.manual_seed(wl.seed + 7 + 1000 * rank)
    dt = -0.125
    stream = torch.cuda.current_stream()
    if wl.extra.get("ends"):
        # both ends: latents of the two modalities, patch projections and output heads
        cv, ca = wl.extra["c_video"], wl.extra["c_audio"]
        ends = make_ends(torch, shape, cv, ca, wl.seed + 2000 + 1000 * rank, dev)
        z0 = torch.randn(shape.n_video * cv + shape.n_audio * ca, generator=gz, device=dev,
                         dtype=torch.float32)
        z = z0.clone()
        zv = z[:shape.n_video * cv].view(shape.n_video, cv)
        za = z[shape.n_video * cv:].view(shape.n_audio, ca)
        rv = torch.zeros(2, shape.n_video, cv, dtype=torch.float32, device=dev)
        ra = torch.zeros(2, shape.n_audio, ca, dtype=torch.float32, device=dev)

        red = wl.extra.get("reduction")

        def step_for(zb):
            zvb = zb[:shape.n_video * cv].view(shape.n_video, cv)
            zab = zb[shape.n_video * cv:].view(shape.n_audio, ca)

            def run(st):
                h3.sample_step(cs, ends, blocks, ids, zvb, zab, rv, ra, None,
                               h3.H3DIT_PASS_FRESH, (1.0, 0.0, 0.0, dt), (1.0, 0.0, 0.0, dt), 0,
                               ws, stream=st, reduction=red)
            return run
    else:
        z0 = torch.randn(N, D, generator=gz, device=dev, dtype=torch.float32)
        z = z0.clone()
        ring = torch.zeros(2, N, D, dtype=torch.float32, device=dev)

        def step_for(zb):
            def run(st):
                h3.denoise_step(cs, blocks, ids, zb, ring, True, (1.0, 0.0, 0.0, dt), 0, ws,
                                stream=st)
            return run

    step_on = step_for(z)

    def step():
        step_on(stream.cuda_stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        z.copy_(z0)
        step()
    torch.cuda.synchronize()
    if h3.sync_status(ws) != 0:
        raise SystemExit("device status error after warm-up")
    barrier()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.3)
    h3.profile_begin(16 * n_blocks * args.steps + 64)
    l0 = h3.launch_count()
    ms, per_step = timed_steps(torch, stream, step, args.steps)
    stages = h3.profile_end()
    launches = h3.launch_count() - l0
    clocks = sampler.stop()
    barrier()
    if h3.sync_status(ws) != 0:
        raise SystemExit("device status error in the timed region")
    ms_max = max_over_ranks(ms, world, dev)

    # end to end through the C ABI with host buffers: every step copies its latents in
    # from pinned host memory, runs, and copies its result back.  Serial: H2D, step, D2H
    # in one stream.  Pipelined (the headline e2e): the steps are independent requests, so
    # two device latent buffers alternate and the copies run on a second stream, each
    # step's H2D and the previous step's D2H overlapping the compute stream.
    z_host = z0.cpu().pin_memory()
    z_back = [torch.empty_like(z_host).pin_memory() for _ in range(2)]
    e2e_ms = e2e_serial_ms = None
    if not args.no_e2e:
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            z.copy_(z_host, non_blocking=True)
            step()
            z_back[0].copy_(z, non_blocking=True)
        torch.cuda.synchronize()
        e2e_serial_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
        assert torch.isfinite(z_back[0]).all().item()
        zb = [z, torch.empty_like(z)]
        runs = [step_for(zb[0]), step_for(zb[1])]
        copy = torch.cuda.Stream()
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(copy):
            zb[0].copy_(z_host, non_blocking=True)
            ev_in[0].record(copy)
        for i in range(args.steps):
            b = i % 2
            stream.wait_event(ev_in[b])
            runs[b](stream.cuda_stream)
            ev_done[b].record(stream)
            with torch.cuda.stream(copy):
                if i + 1 < args.steps:  # buffer b ^ 1: its previous D2H is earlier in this stream
                    zb[b ^ 1].copy_(z_host, non_blocking=True)
                    ev_in[b ^ 1].record(copy)
                copy.wait_event(ev_done[b])
                z_back[b].copy_(zb[b], non_blocking=True)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
        assert all(torch.isfinite(t).all().item() for t in z_back)

    # the same step captured once into a CUDA graph and replayed
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step_on(side.cuda_stream)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        c0 = h3.launch_count()
        with torch.cuda.graph(g):
            step_on(torch.cuda.current_stream().cuda_stream)
        g_launches = h3.launch_count() - c0
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        barrier()
        g_ms, g_per = timed_steps(torch, stream, g.replay, args.steps)
        if h3.sync_status(ws) != 0:
            raise SystemExit("device status error in the graph replays")
        g_ms = max_over_ranks(g_ms, world, dev)
        graph = {"value": job_rows_per_s(N * n_blocks * args.steps, world, g_ms),
                 "ms_per_step": g_ms / args.steps, "ms_per_step_median": median(g_per),
                 "launches_per_step": int(g_launches),
                 "how": "one step captured into a CUDA graph, replayed per step"}
        del g

    ties = None
    if not args.no_ties and rank == 0:
        xr = z0.view(-1)[:N * D].view(N, D).to(torch.bfloat16) if not wl.extra.get("ends") \
            else torch.randn(N, D, generator=gz, device=dev).to(torch.bfloat16)
        ties = block_near_ties(h3, torch, shape, blocks[0], xr, dev)

    if rank != 0:
        return None
    K = args.steps
    rows_blocks = N * n_blocks * K * world
    value = job_rows_per_s(N * n_blocks * K, world, ms_max)
    # the shape each block position runs at (token reduction shrinks the video rows)
    shapes = block_shapes(shape, n_blocks, wl.extra.get("reduction"))
    step_flops = sum(sum(block_flops(sb)) for sb in shapes)
    pk, pk_kind = peaks()
    peak_tc = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    achieved_total = step_flops * K / (ms_max / 1e3) / 1e12
    clk_peak = per_clock_peak(props.multi_processor_count, (clocks or {}).get("sm_mhz"))
    roofline, kernels = dominant_kernel(shape, shapes, stages, K, wl.name, clk_peak)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_max / K,
        "ms_per_step_median": median(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": forward_config(wl, n_blocks, world),
        "s_per_forward": ms_max / K / 1e3 * (50 / n_blocks),
        "tc_frac_of_peak": achieved_total / peak_tc,
        "tc_frac_of_peak_per_clock": achieved_total / clk_peak if clk_peak else None,
        "achieved_tflops": achieved_total,
        "roofline": roofline,
        "stages_ms_per_step": {k: v[0] / K for k, v in stages.items()},
        "kernels": kernels,
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if graph is not None:
        out["graph"] = graph
    if ties is not None:
        out["near_ties"] = ties
    if e2e_ms is not None:
        out["e2e"] = {"value": rows_blocks / (e2e_ms / 1e3), "unit": UNIT,
                      "h2d_bytes_per_step": z.numel() * 4, "d2h_bytes_per_step": z.numel() * 4,
                      "mode": "pipelined: independent steps, two latent buffers, copies on a "
                              "second stream overlapping the neighbouring steps' compute",
                      "serial": {"value": rows_blocks / (e2e_serial_ms / 1e3),
                                 "mode": "H2D, step, D2H in one stream"}}
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(shape)
        out["cpu_baseline"].pop("s_per_block")
    return out


def fresh_schedule(n_steps, reuse):
    """Passes that run the model: every reuse-th pass and the last one."""
    return [i % reuse == 0 or i == n_steps - 1 for i in range(n_steps)]


def run_loop(args, rank, world, local_rank):
    """The 20-step denoising loop at 4,096 rows: 45 of 50 blocks kept by layer thinning,
    velocity reuse 2 (11 fresh passes), plus a top-k density sweep of one block."""
    import numpy as np
    import torch

    import audio_diffusion_transformer_gb300 as h3
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = S.workload_by_name(args.workload)
    shape = wl.shape
    N, D = shape.n_rows, shape.hidden
    n_steps, reuse, keep = wl.extra["steps"], wl.extra["reuse"], wl.extra["keep"]
    cs = h3.make_shape(shape)
    ws_bytes = max(h3.workspace_bytes(h3.make_shape(shape.with_(topk=k)))
                   for k in [shape.topk] + list(wl.extra["topk_sweep"]))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    blocks = make_blocks(torch, shape, wl.n_blocks, wl.seed + 1000 * rank, dev)
    mods = np.stack([b["mod"].cpu().numpy() for b in blocks])
    ids = h3.select_blocks(mods, keep)
    gz = torch.Generator(device=dev)
    gz.manual_seed(wl.seed + 7 + 1000 * rank)
    z0 = torch.randn(N, D, generator=gz, device=dev, dtype=torch.float32)
    z = z0.clone()
    ring = torch.zeros(2, N, D, dtype=torch.float32, device=dev)
    sig = [1.0 - i / n_steps for i in range(n_steps + 1)]
    dt = -1.0 / n_steps
    fresh = fresh_schedule(n_steps, reuse)
    stream = torch.cuda.current_stream()

    def eager_loop(st=None):
        st = stream.cuda_stream if st is None else st
        z.copy_(z0)
        nf, fs = 0, []
        for i in range(n_steps):
            if fresh[i]:
                h3.denoise_step(cs, blocks, ids, z, ring, True, (sig[i], 0.0, 0.0, dt), nf, ws,
                                stream=st)
                nf += 1
                fs.append(sig[i])
            else:
                sb = fs[-2] if len(fs) > 1 else fs[-1]
                h3.denoise_step(cs, blocks, ids, z, ring, False, (sig[i], fs[-1], sb, dt), nf,
                                ws, stream=st)

    loop = eager_loop
    graph_launches = None
    if args.graph:
        # the whole loop (~4,500 launches) captured once into a CUDA graph and replayed
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            eager_loop(side.cuda_stream)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        c0 = h3.launch_count()
        with torch.cuda.graph(graph):
            eager_loop(torch.cuda.current_stream().cuda_stream)
        graph_launches = h3.launch_count() - c0
        loop = graph.replay

    for _ in range(args.warmup):
        loop()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler()
    sampler.start()
    time.sleep(0.3)
    l0 = h3.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        loop()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = h3.launch_count() - l0
    if graph_launches is not None:  # replays launch the captured kernels without the host
        launches = graph_launches * args.steps
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    if h3.sync_status(ws) != 0:
        raise SystemExit("device status error in the timed region")
    ms = max_over_ranks(ms, world, dev)
    # stage times from one separately profiled pass: at 4,096 rows the loop is
    # launch-heavy and per-stage events in the timed region would slow it by ~3%
    h3.profile_begin(16 * n_steps * len(ids) + 64 * n_steps)
    eager_loop()
    torch.cuda.synchronize()
    stages = h3.profile_end()
    # end to end: H2D of the latents, the loop, D2H of the result, every timed step
    e2e_ms = None
    if not args.no_e2e:
        z_host = z0.cpu().pin_memory()
        z_back = torch.empty_like(z_host).pin_memory()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            z0.copy_(z_host, non_blocking=True)
            loop()
            z_back.copy_(z, non_blocking=True)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
    n_fresh = sum(fresh)
    block_evals = n_fresh * len(ids)
    # top-k density sweep: one block of this shape per k, rows/s per block
    sweep = {}
    x0 = torch.randn(N, D, generator=gz, device=dev, dtype=torch.float32).to(torch.bfloat16)
    for k in wl.extra["topk_sweep"]:
        csk = h3.make_shape(shape.with_(topk=k))
        x = x0.clone()
        for _ in range(3):
            h3.block_forward(csk, blocks[0], x, ws, stream=stream.cuda_stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for r in range(10):
            h3.block_forward(csk, blocks[r % len(blocks)], x, ws, stream=stream.cuda_stream)
        b.record(stream)
        torch.cuda.synchronize()
        t_ms = a.elapsed_time(b) / 10
        gf, af = block_flops(shape.with_(topk=k))
        sweep[str(k)] = {"rows_per_s": N / (t_ms / 1e3), "ms_per_block": t_ms,
                         "attention_gflop": af / 1e9, "tflops": (gf + af) / (t_ms / 1e3) / 1e12}
    if rank != 0:
        return None
    pk, pk_kind = peaks()
    gf, af = block_flops(shape)
    achieved = block_evals * (gf + af) * args.steps / (ms / 1e3) / 1e12
    roofline, kernels = dominant_kernel(shape, [shape], stages, 1, wl.name, calls=block_evals)
    roofline["measured"] = "one profiled pass after the timed region"
    extra = {"roofline": roofline, "kernels": kernels,
             "stages_ms_per_step": {k: v[0] for k, v in stages.items()}}
    if e2e_ms is not None:
        extra["e2e"] = {"value": job_rows_per_s(N * block_evals * args.steps, world, e2e_ms),
                        "unit": UNIT, "h2d_bytes_per_step": N * D * 4,
                        "d2h_bytes_per_step": N * D * 4}
    return dict(extra, **{
        "metric": METRIC, "value": job_rows_per_s(N * block_evals * args.steps, world, ms),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "n_rows": N, "hidden": D, "heads": shape.heads,
                   "head_dim": shape.head_dim, "topk": shape.topk, "denoise_steps": n_steps,
                   "reuse": reuse, "fresh_passes": n_fresh, "blocks_kept": len(ids),
                   "blocks_total": wl.n_blocks, "kept_ids": ids,
                   "parallelism": f"replicas x{world}",
                   "launch": "one CUDA graph per loop" if args.graph else "eager",
                   "l2": "inputs larger than L2 (45 blocks x 113 MB of weights per pass)"},
        "tc_frac_of_peak": achieved / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
        "achieved_tflops": achieved, "topk_sweep": sweep, "gpu_launches": int(launches),
        "clocks": clocks,
    })


WORKLOAD_ALIASES = {"routed_attention_1024": "attn_tiny_1024"}


def attention_flops(s):
    """Algorithmic attention flops of one routed-attention call (4 d per query-key pair)."""
    return block_flops(s)[1]


def run_attention_only(args, rank, world, local_rank):
    """h3dit_routed_attention alone on the 1,024-row case (4 heads x 64, 16 tiles of 64,
    N(0,1) Q/K/V and gate from seed): top-k 4 with the pooled branch (the line's value)
    and top-k 16 (every tile: dense attention).  Each timed call is bracketed by events
    on its stream and preceded by an L2 flush (a 256 MB write) outside the brackets."""
    import numpy as np
    import torch

    import audio_diffusion_transformer_gb300 as h3
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = S.ATTN_TINY
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    inp = S.attention_inputs(wl.shape, wl.seed + 1000 * rank)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).to(dev)

    q, k, v, g = (to_dev(inp[n]) for n in ("q", "k", "v", "gate"))
    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(getattr(props, "pci_bus_id", None))
    lines = {}
    for topk in (wl.shape.topk, 16):
        shp = wl.shape.with_(topk=topk)
        cs = h3.attn_shape(shp)
        ws = torch.zeros(h3.workspace_bytes(cs), dtype=torch.uint8, device=dev)
        tv = shp.n_video_tiles
        kk = min(topk, tv)
        out = torch.empty(shp.n_rows, shp.attn_width, dtype=torch.bfloat16, device=dev)
        idx = torch.empty(shp.heads, tv, kk, dtype=torch.int32, device=dev)
        sc = torch.empty(shp.heads, tv, tv, dtype=torch.float32, device=dev)

        def call():
            h3.routed_attention(cs, q, k, v, g, out, ws, idx=idx, scores=sc,
                                stream=stream.cuda_stream)

        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        if topk == wl.shape.topk:
            sampler.start()
            time.sleep(0.2)
        h3.profile_begin(4 * args.steps + 8)
        l0 = h3.launch_count()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
        stages = h3.profile_end()
        launches = h3.launch_count() - l0
        if h3.sync_status(ws) != 0:
            raise SystemExit("device status error in the timed region")
        per = [a.elapsed_time(b) for a, b in evs]
        att_ms = stages["attention"][0] / max(stages["attention"][1], 1)
        fl = attention_flops(shp)
        lines[topk] = {"ms_per_call": sum(per) / len(per), "ms_per_call_median": median(per),
                       "rows_per_s": shp.n_rows / (sum(per) / len(per) / 1e3),
                       "attention_kernel_ms": att_ms,
                       "router_ms": stages["router"][0] / max(stages["router"][1], 1),
                       "attention_gflop": fl / 1e9,
                       "attention_tflops": fl / (att_ms / 1e3) / 1e12 if att_ms else None,
                       "gpu_launches": int(launches),
                       "near_ties": near_tie_audit(sc.cpu().numpy(), idx.cpu().numpy(), kk)}
        if topk == wl.shape.topk:
            clocks = sampler.stop()
            # end to end: H2D of q, k, v, gate from pinned memory, the call, D2H of out
            hq, hk, hv, hg = (t.cpu().pin_memory() for t in (q, k, v, g))
            ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            dq, dk, dv, dg = (torch.empty_like(t) for t in (q, k, v, g))
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(args.steps):
                for d_, h_ in ((dq, hq), (dk, hk), (dv, hv), (dg, hg)):
                    d_.copy_(h_, non_blocking=True)
                h3.routed_attention(cs, dq, dk, dv, dg, out, ws, stream=stream.cuda_stream)
                ho.copy_(out, non_blocking=True)
            torch.cuda.synchronize()
            e2e_s = (time.perf_counter() - t0) / args.steps
            lines[topk]["e2e"] = {"value": shp.n_rows / e2e_s, "unit": UNIT,
                                  "h2d_bytes_per_step": sum(t.numel() * 2 for t in (q, k, v, g)),
                                  "d2h_bytes_per_step": out.numel() * 2}
    if rank != 0:
        return None
    main = lines[wl.shape.topk]
    pk, pk_kind = peaks()
    peak_tc = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    value = main["rows_per_s"] * world
    bytes_moved = (3 * wl.shape.heads * wl.shape.n_rows * wl.shape.head_dim * 2
                   + 2 * wl.shape.n_rows * wl.shape.attn_width * 2)
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": main["ms_per_call"],
           "ms_per_step_median": main["ms_per_call_median"], "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": wl.name, "n_rows": wl.shape.n_rows, "heads": wl.shape.heads,
                      "head_dim": wl.shape.head_dim, "tiles": wl.shape.n_video_tiles,
                      "topk": wl.shape.topk, "pooled": True, "parallelism": f"replicas x{world}",
                      "l2": "L2 flushed (256 MB write) before every timed call",
                      "step": "one h3dit_routed_attention call (router + attention)"},
           "roofline": {"bound": "tensor", "kernel": "attention",
                        "achieved": main["attention_tflops"], "peak": peak_tc,
                        "peak_kind": f"bf16 sustained, {pk_kind}", "unit": "TFLOP/s",
                        "frac": (main["attention_tflops"] or 0) / peak_tc, "traffic": None,
                        "note": "latency-bound: 32 work units for 152 SMs; "
                                f"{bytes_moved / 1e6:.1f} MB of q, k, v, gate and output"},
           "topk_4": main, "dense_topk_16": lines[16],
           "near_ties": main["near_ties"], "gpu_launches": main["gpu_launches"],
           "clocks": clocks, "e2e": main["e2e"]}
    if not args.no_cpu_baseline and world == 1:
        from oracle import ctime
        qf, kf, vf, gf = (S.bf16_bits_to_f64(inp[n]).astype(np.float32)
                          for n in ("q", "k", "v", "gate"))
        att = ctime.Attention(wl.shape, qf, kf, vf, gf)
        att.run()
        reps = 0
        t0 = time.perf_counter()
        while reps < 3 or time.perf_counter() - t0 < 2.0:
            att.run()
            reps += 1
        t = (time.perf_counter() - t0) / reps
        out["cpu_baseline"] = {"value": wl.shape.n_rows / t, "unit": UNIT,
                               "cores": ctime.threads(), "kind": "oracle fp32, measured full call",
                               "sample": f"the float32 C oracle's router + attention + pooled "
                                         f"mix on the same inputs, {reps} calls averaged"}
    return out


def run_reference_attention(args, world):
    """CPU oracle arm of the 1,024-row attention line: the float32 C oracle's router,
    attention and pooled mix on the same inputs, every step timed."""
    import numpy as np

    from oracle import ctime
    wl = S.ATTN_TINY
    inp = S.attention_inputs(wl.shape, wl.seed)
    qf, kf, vf, gf = (S.bf16_bits_to_f64(inp[n]).astype(np.float32)
                      for n in ("q", "k", "v", "gate"))
    att = ctime.Attention(wl.shape, qf, kf, vf, gf)
    for _ in range(args.warmup):
        att.run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        att.run()
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = wl.shape.n_rows * args.steps / tot
    desc = "float32 C oracle: router, attention and pooled mix of the 1,024-row call"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3,
            "ms_per_step_median": median(times) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "n_rows": wl.shape.n_rows, "heads": wl.shape.heads,
                       "head_dim": wl.shape.head_dim, "tiles": wl.shape.n_video_tiles,
                       "topk": wl.shape.topk, "pooled": True,
                       "parallelism": f"replicas x{world}",
                       "l2": "L2 flushed (256 MB write) before every timed call",
                       "step": "one h3dit_routed_attention call (router + attention)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": ctime.threads(),
                             "kind": "oracle fp32, measured full call", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_reference(args, rank, world):
    """The CPU oracle arm: each step runs the float32 C oracle on the same workload shape,
    on all host cores -- the whole block when a step fits about four seconds, else a
    uniform 1/s sample chosen from a calibration call -- and every step is timed."""
    if rank != 0:
        return None
    from oracle import ctime
    if S.workload_by_name(args.workload) is S.ATTN_TINY:
        return run_reference_attention(args, world)
    wl, n_blocks = workload(args.workload)
    blk, x, s = cpu_block(wl.shape)
    sample, est_full = cpu_sample_plan(blk, x, s.n_rows, 4.0)
    rows = sampled_rows(s.n_rows, sample)
    for _ in range(args.warmup):
        time_cpu_block(blk, x, sample)
    times = [time_cpu_block(blk, x, sample) for _ in range(args.steps)]
    tot = sum(times)
    value = rows * args.steps / tot
    s_block = tot / args.steps * s.n_rows / rows
    desc = sample_desc(s, sample, s.n_rows)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": tot / args.steps * 1e3,
           "ms_per_step_median": sorted(times)[len(times) // 2] * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic", "config": forward_config(wl, n_blocks, world),
           "step": desc,
           "s_per_block": s_block,
           "s_per_forward": s_block * 50,
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": ctime.threads(),
                            "kind": "oracle fp32, measured " + ("full block" if sample == 1
                                                                else f"1/{sample} sample"),
                            "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    if sample > 1:
        out["extrapolated_from"] = (f"1/{sample} sample per step: s_per_block and "
                                    f"s_per_forward scale the measured step time by "
                                    f"{s.n_rows}/{rows} rows (and x50 blocks)")
    else:
        out["extrapolated_from"] = "s_per_forward = 50 x the measured block"
    if s is not wl.shape:
        out["slice_tiles"] = "cube layout timed with 64-row slice tiles of the same sizes"
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="forward50_15435_d5120")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay arm of a forward line")
    ap.add_argument("--no-ties", action="store_true", help="skip the near-tie audit")
    ap.add_argument("--graph", action="store_true",
                    help="loop workload: capture the loop into a CUDA graph and replay it")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    args.workload = WORKLOAD_ALIASES.get(args.workload, args.workload)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        if S.workload_by_name(args.workload) is S.LOOP_4K:
            out = run_loop(args, rank, world, local_rank)
        elif S.workload_by_name(args.workload) is S.ATTN_TINY:
            out = run_attention_only(args, rank, world, local_rank)
        else:
            out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()

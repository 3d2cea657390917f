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

--impl reference times the CPU oracle (float64, numpy) on a bounded sample of
the same workload on this host's cores.  Multi-GPU runs are independent
replicas (one per rank, no data-path collective).
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
_SAMPLE_INPUTS = {}


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


def oracle_block_sample(shape, rng_seed=0):
    """Times the oracle on a bounded sample of one block of ``shape`` and scales it
    to the whole block.  Returns (seconds per block, description)."""
    import numpy as np

    import oracle as O
    s = shape
    N, D, A, F, H, d = s.n_rows, s.hidden, s.attn_width, s.mlp_width, s.heads, s.head_dim
    R = min(N, 2048)   # rows through the row-local stages
    HS = min(H, 12)    # heads through the router and attention
    key = (N, D, A, F, H, d, s.mlp, rng_seed)
    if key not in _SAMPLE_INPUTS:  # drawn once per process; only the oracle's work is timed
        rng = np.random.default_rng(rng_seed)
        _SAMPLE_INPUTS[key] = (
            {"w_qkvg": O.bf16(rng.standard_normal((4 * A, D)) * 0.02),
             "b_qkvg": O.bf16(rng.standard_normal(4 * A) * 0.02),
             "w_o": O.bf16(rng.standard_normal((D, A)) * 0.02), "b_o": np.zeros(D),
             "w1": O.bf16(rng.standard_normal((2 * F if s.mlp == "swiglu" else F, D)) * 0.02),
             "b1": np.zeros(2 * F if s.mlp == "swiglu" else F),
             "w2": O.bf16(rng.standard_normal((D, F)) * 0.02), "b2": np.zeros(D),
             "mod": rng.standard_normal((6, D)) * 0.1},
            O.bf16(rng.standard_normal((R, D))),
            [O.bf16(rng.standard_normal((HS, N, d))) for _ in range(3)])
    w, x, (Q, K, V) = _SAMPLE_INPUTS[key]
    # row-local stages on R rows
    t0 = time.perf_counter()
    h = O.rms_modulate(x, w["mod"][0], w["mod"][1])
    qkvg = O.bf16(O.linear(h, w["w_qkvg"], w["b_qkvg"]))
    O.qkv_heads(qkvg, H, d, np.ones(d), np.ones(d))
    o = O.bf16(qkvg[:, :A])
    x1 = O.bf16(x + w["mod"][2] * O.linear(o, w["w_o"], w["b_o"]))
    h2 = O.rms_modulate(x1, w["mod"][3], w["mod"][4])
    u = O.mlp_inner(h2, w, s.mlp)
    O.bf16(x1 + w["mod"][5] * O.linear(u, w["w2"], w["b2"]))
    t_rows = (time.perf_counter() - t0) * N / R
    # router over all tiles, attention for a sample of query tiles of a few heads
    hs = HS
    t0 = time.perf_counter()
    mq = O.tile_means(Q, s.n_prefix, s.n_video)
    mk = O.tile_means(K, s.n_prefix, s.n_video)
    mv = O.tile_means(V, s.n_prefix, s.n_video)
    Sc = O.tile_scores(mq, mk)
    idx = O.topk_select(Sc, s.topk)
    O.pooled_branch(Sc, mv, d)
    t_router = (time.perf_counter() - t0) * H / hs
    tv = s.n_video_tiles
    vt = [(h, i) for h in range(hs) for i in range(0, tv, max(1, tv // 12))][:12 * hs]
    t0 = time.perf_counter()
    O.routed_attention(Q, K, V, s.n_prefix, s.n_video, idx, tiles=vt)
    t_vid = (time.perf_counter() - t0) * (H * tv) / len(vt)
    t_pre = 0.0
    n_chunks = 0
    if s.n_prefix:
        t0 = time.perf_counter()
        n_chunks = min(2, (s.n_prefix + 63) // 64)
        pre_rows = min(s.n_prefix, 64 * n_chunks)  # prefix query rows attended per head
        for h in range(hs):
            for c in range(n_chunks):
                O.attend(Q[h, 64 * c:min(64 * c + 64, s.n_prefix)], K[h], V[h],
                         1.0 / math.sqrt(d))
        t_pre = (time.perf_counter() - t0) * (H * s.n_prefix) / (hs * pre_rows)
    total = t_rows + t_router + t_vid + t_pre
    pre = (f" and {hs * n_chunks} prefix chunks of up to 64 rows "
           f"(x{H * s.n_prefix / (hs * pre_rows):.3g})" if n_chunks else "")
    desc = (f"one block of the {N}-row shape, float64 oracle: row-local stages on {R} rows "
            f"(x{N / R:.3g}), router on {hs} of {H} heads (x{H / hs:.3g}), attention on "
            f"{len(vt)} video query tiles (x{H * tv / len(vt):.3g}){pre}; scaled to the whole "
            f"block")
    return total, desc


def blas_threads():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count() or 1


def cpu_baseline(shape, samples=1):
    best = None
    desc = ""
    for _ in range(samples):
        t, desc = oracle_block_sample(shape)
        best = t if best is None else min(best, t)
    return {"value": shape.n_rows / best, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": desc, "s_per_block": best}


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


def dominant_kernel(shape, shapes, stages, K, workload_name):
    """Roofline of the kernel with the largest stage time, from the live stage records
    (ms, launches); achieved = its algorithmic flops / its time.  Also per-kernel rates."""
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
    n_launch = sum(stages[s_][1] for s_ in groups[dom])
    flops = sum(sf[s_] * stages[s_][1] for s_ in groups[dom])
    kernel = "attention" if dom == "attention" else "gemm"
    roofline = {"bound": "tensor", "kernel": dom,
                "achieved": flops / (g_ms[dom] / 1e3) / 1e12, "peak": peak_tc,
                "peak_kind": f"bf16 sustained, {pk_kind}", "unit": "TFLOP/s",
                "traffic": recorded_traffic(kernel, dom, workload_name),
                "launch_ms": g_ms[dom] / max(n_launch, 1), "launches": n_launch}
    roofline["frac"] = roofline["achieved"] / peak_tc
    kernels = {}
    for g, st in groups.items():
        fl = sum(sf[s_] * stages[s_][1] for s_ in st)
        kernels[g] = {"ms_per_step": g_ms[g] / K,
                      "tflops": fl / (g_ms[g] / 1e3) / 1e12 if g_ms[g] > 0 else None}
    return roofline, kernels


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

        def step():
            h3.sample_step(cs, ends, blocks, ids, zv, za, rv, ra, None, h3.H3DIT_PASS_FRESH,
                           (1.0, 0.0, 0.0, dt), (1.0, 0.0, 0.0, dt), 0, ws,
                           stream=stream.cuda_stream, reduction=red)
    else:
        z0 = torch.randn(N, D, generator=gz, device=dev, dtype=torch.float32)
        z = z0.clone()
        ring = torch.zeros(2, N, D, dtype=torch.float32, device=dev)

        def step():
            h3.denoise_step(cs, blocks, ids, z, ring, True, (1.0, 0.0, 0.0, dt), 0, ws,
                            stream=stream.cuda_stream)

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
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except AttributeError:
        pass
    sampler = ClockSampler(bus)
    sampler.start()
    time.sleep(0.3)
    h3.profile_begin(16 * n_blocks * args.steps + 64)
    l0 = h3.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    stages = h3.profile_end()
    launches = h3.launch_count() - l0
    clocks = sampler.stop()
    barrier()
    ms = e0.elapsed_time(e1)
    if h3.sync_status(ws) != 0:
        raise SystemExit("device status error in the timed region")
    ms_max = max_over_ranks(ms, world, dev)

    # end to end through the C ABI with host buffers: H2D z, the step, D2H z
    z_host = z0.cpu().pin_memory()
    z_back = torch.empty_like(z_host).pin_memory()
    e2e_ms = None
    if not args.no_e2e:
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            z.copy_(z_host, non_blocking=True)
            step()
            z_back.copy_(z, non_blocking=True)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
        assert torch.isfinite(z_back).all().item()

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
    roofline, kernels = dominant_kernel(shape, shapes, stages, K, wl.name)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": forward_config(wl, n_blocks, world),
        "s_per_forward": ms_max / K / 1e3 * (50 / n_blocks),
        "tc_frac_of_peak": achieved_total / peak_tc,
        "achieved_tflops": achieved_total,
        "roofline": roofline,
        "stages_ms_per_step": {k: v[0] / K for k, v in stages.items()},
        "kernels": kernels,
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if e2e_ms is not None:
        out["e2e"] = {"value": rows_blocks / (e2e_ms / 1e3), "unit": UNIT,
                      "h2d_bytes_per_step": z.numel() * 4, "d2h_bytes_per_step": z.numel() * 4}
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
    roofline, kernels = dominant_kernel(shape, [shape], stages, 1, wl.name)
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


def run_reference(args, rank, world):
    if rank != 0:
        return None
    wl, n_blocks = workload(args.workload)
    shape = wl.shape
    for _ in range(args.warmup):
        oracle_block_sample(shape)
    tot = 0.0
    desc = ""
    for _ in range(args.steps):
        t, desc = oracle_block_sample(shape)
        tot += t
    value = shape.n_rows * args.steps / tot
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3 * n_blocks, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": forward_config(wl, n_blocks, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="forward50_15435_d5120")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="loop workload: capture the loop into a CUDA graph and replay it")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
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
        else:
            out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()

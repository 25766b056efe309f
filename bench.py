"""Benchmark of the MpFA QK4PV8 attention forward on GB300.

One step = the whole prefill hot path on the largest single-GPU workload,
the Qwen3-14B attention shape at 128K (B=1, 40 query / 8 KV heads, d=128,
N=131072, causal): online NVFP4/FP8 quantization of Q, K, V
(mpfa_quantize_qkv) followed by the prefill kernel (mpfa_prefill), on
synthetic inputs resident in HBM.  ``value`` is the algorithmic attention
TFLOP/s of that step (512 FLOP per visible (query, key) pair: 256 for QK^T in
FP4, 256 for PV in FP8).  The inputs (1.9 GB of bf16) are larger than L2,
and L2 is also flushed (a 512 MB write) before every timed step.

The same JSON line carries:
  roofline      prefill kernel vs the FP4/FP8 tensor-pipe roofline
  prefill_other the other prefill workloads (Llama-3.1-8B shape at 16K, the
                B1/S4096/H24 and B1/S8192/H64 grid), each with its roofline
  decode        split-KV decode on B=64 x 32K and on B=64 x U[4K, 64K]
                cached tokens: KV GB/s vs HBM
  e2e           the step through the C ABI with host buffers (pinned H2D of
                bf16 Q/K/V, D2H of O and LSE) inside the timed region
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
  clocks        nvidia-smi samples taken during the timed region

``--impl reference`` times the CPU oracle instead (the reference arm).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import mpfa_inputs as mi  # noqa: E402

METRIC = "prefill attention TFLOP/s & decode KV GB/s on 1 GB300, % of FP4/FP8/HBM roofline"
HEADLINE = "qwen14b_n128k_causal"
OTHER_PREFILL = ("llama8b_n16k_causal", "b1_s4096_h24", "b1_s8192_h64")
DECODES = ("decode_b64_l32k", "decode_b64_l4k_64k")
FLOP_PER_PAIR = 512
KV_BYTES_PER_TOKEN = 64 + 8 + 128   # K codes + K block scales + V codes, per KV head
T_TERMS = 2


def prefill_algo_bytes(cfg, T=T_TERMS) -> int:
    """prefill_kernel inputs and outputs per launch: Q codes + block scales,
    rank-one terms, K codes + scales, V codes, O (bf16) and LSE."""
    return (cfg.B * cfg.N * (cfg.Hq * (64 + 8 + 128 * 2 + 4) + cfg.Hkv * (64 + 8 + 128))
            + cfg.B * cfg.Hq * (cfg.N // 128) * T * 72)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        """Start sampling; returns once the first sample has arrived (or after
        a few seconds), so that the timed region that follows is covered."""
        import threading
        self.lines = []
        first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader(proc=self.proc):
            for line in proc.stdout:
                self.lines.append(line)
                first.set()
            first.set()
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        first.wait(5.0)
        self.skip = len(self.lines)     # samples taken before the timed region

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)
        sm, mx, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[self.skip:]:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) of `kernel` on `workload` from the
    ncu figures in profiles/traffic.json, or None when the kernel's sources
    have changed since the counters were taken (sha256 of the listed files)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    csrc = os.path.join(ROOT, "flashattention_mpfa_quantize_gb300", "csrc")
    with open(path) as f:
        doc = json.load(f)
    for row in doc.get("kernels", []):
        if row.get("kernel") != kernel or row.get("workload") != workload:
            continue
        h = hashlib.sha256()
        try:
            for src in row["sources"]:
                with open(os.path.join(csrc, src), "rb") as fh:
                    h.update(fh.read())
        except OSError:
            return None
        if h.hexdigest()[:16] != row["sha16"]:
            return None
        return int(round((int(row["read"]) + int(row["write"])) * float(row.get("scale", 1.0))))
    return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """Largest x over all ranks (x itself without a process group).  The
    tensor lives on `device` for NCCL and on the host for gloo."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    on = "cpu" if dist.get_backend() == "gloo" or device is None else device
    t = torch.tensor([float(x)], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, ms_local: float, world: int, device=None):
    """Whole-job rate of replicas that each process `units_per_rank` units:
    the units of all ranks over the slowest rank's time.  Returns (rate in
    units/s, the max-over-ranks ms)."""
    ms = max_over_ranks(ms_local, device)
    return world * units_per_rank / (ms * 1e-3), ms


# ----------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------

def _host_f32(x):
    import numpy as np
    return x if isinstance(x, np.ndarray) else x.float().cpu().numpy()


def oracle_scales(cfg, Qn, Kn, Vn):
    """Whole-tensor statistics the codes depend on (tensor scales of Q' with
    the rank-one smoothing, K and V).  Returns ((s_q, s_k, s_v), seconds)."""
    import numpy as np

    import oracle as orc
    t0 = time.perf_counter()
    amax_q = np.float32(0)
    for b in range(cfg.B):
        for h in range(cfg.Hq):
            qb, qp = orc.block_means(np.ascontiguousarray(Qn[b, :, h, :]), 128)
            amax_q = max(amax_q, np.float32(np.abs(qp).max()), np.float32(np.abs(qb).max()))
    s = (orc.tensor_scale(amax_q, 2688.0), orc.tensor_scale(np.abs(Kn).max(), 2688.0),
         orc.tensor_scale(np.abs(Vn).max(), 448.0))
    return s, time.perf_counter() - t0


def oracle_heads(cfg, Qn, Kn, Vn, scales, rows_per_head, heads):
    """Codes of the sampled heads and the emulated forward of sampled query
    rows (spread over the sequence, full causal key range each).
    Returns (flops, seconds, rows)."""
    import numpy as np

    import oracle as orc
    g = cfg.Hq // cfg.Hkv
    s_q, s_k, s_v = scales
    t0 = time.perf_counter()
    flops = 0
    n = cfg.N
    rows = np.unique(np.linspace(0, n - 1, rows_per_head).astype(np.int64))
    for (b, h) in heads:
        hk = h // g
        qb, qp = orc.block_means(np.ascontiguousarray(Qn[b, :, h, :]), 128)
        qc, qs = orc.nvfp4_quantize(qp, s_q)
        tc, ts = orc.rank_one_terms(qb, s_q, T_TERMS)
        kc, ks = orc.nvfp4_quantize(np.ascontiguousarray(Kn[b, :, hk, :]), s_k)
        vc = orc.fp8_quantize(np.ascontiguousarray(Vn[b, :, hk, :]), s_v)
        qz = dict(qc=qc[None, None], qs=qs[None, None], qbc=tc[None, None], qbs=ts[None, None],
                  s_q=s_q)
        kz = dict(kc=kc[None, None], ks=ks[None, None], s_k=s_k)
        vz = dict(vc=vc[None, None], s_v=s_v)
        orc.prefill_emulate(qz, kz, vz, causal=cfg.causal, heads=[(0, 0)], rows=rows)
        flops += FLOP_PER_PAIR * int((rows + 1).sum() if cfg.causal else rows.size * n)
    return flops, time.perf_counter() - t0, rows.size


def oracle_sample(cfg, Q, K, V, rows_per_head, heads):
    """Time the CPU oracle on a bounded sample of the prefill workload: the
    whole-tensor statistics, the codes of the sampled heads and the emulated
    forward of the sampled rows.  Returns (tflops, seconds, description,
    threads)."""
    import oracle as orc
    Qn, Kn, Vn = _host_f32(Q), _host_f32(K), _host_f32(V)
    scales, t_s = oracle_scales(cfg, Qn, Kn, Vn)
    flops, t_h, nrows = oracle_heads(cfg, Qn, Kn, Vn, scales, rows_per_head, heads)
    dt = t_s + t_h
    desc = (f"{len(heads)} heads x {nrows} query rows of {cfg.name} (full causal key "
            f"range each), incl. whole-tensor statistics ({t_s:.1f} s) and per-head "
            f"quantization")
    return flops / dt / 1e12, dt, desc, orc.num_threads()


REFERENCE_BUDGET_S = 90.0   # oracle time of a whole --impl reference run


def run_reference(args):
    """The CPU oracle as it stands on the headline workload.  The whole-tensor
    statistics are computed once per run (their time counts, spread over the
    steps); each step then quantizes a sampled head and emulates sampled
    query rows, sized from two calibration samples so the timed work takes
    about REFERENCE_BUDGET_S in all, whatever --steps is."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    cfg = mi.PREFILL[args.workload]
    Q, K, V = mi.prefill_inputs(cfg, "cpu", 0)
    Qn, Kn, Vn = Q.float().numpy(), K.float().numpy(), V.float().numpy()
    del Q, K, V
    for _ in range(max(args.warmup, 1)):
        oracle_heads(cfg, Qn, Kn, Vn, (1.0, 1.0, 1.0), 2, ((0, 0),))
    scales, t_scales = oracle_scales(cfg, Qn, Kn, Vn)
    heads = ((0, 0),)
    t_small = oracle_heads(cfg, Qn, Kn, Vn, scales, 2, heads)[1]
    t_big = oracle_heads(cfg, Qn, Kn, Vn, scales, 34, heads)[1]
    per_row = max((t_big - t_small) / 32.0, 1e-6)
    target = max(REFERENCE_BUDGET_S - t_scales, 1.0) / max(args.steps, 1)
    rows = int(max(2, min(256, 2 + (target - t_small) / per_row)))
    flops_all, t_all = 0, t_scales
    times = []
    nrows = 0
    for i in range(args.steps):
        h = (0, (9 * i) % cfg.Hq)
        f, dt, nrows = oracle_heads(cfg, Qn, Kn, Vn, scales, rows, (h,))
        flops_all += f
        t_all += dt
        times.append(dt + t_scales / max(args.steps, 1))
    value = flops_all / t_all / 1e12
    thr = orc.num_threads()
    desc = (f"per step 1 head x {nrows} query rows of {cfg.name} (full causal key range "
            f"each) incl. that head's quantization; whole-tensor statistics once per run "
            f"({t_scales:.2f} s, counted)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (emulated nvfp4/fp8 codes)",
            "data": "synthetic", "config": {"workload": cfg.name, "sample": desc},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def prefill_roofline(cfg, pre_ms, peaks, pv4=False):
    """prefill_kernel against the FP4 QK^T + FP8 PV tensor-pipe roofline: the
    measured bf16 peak times the nominal dense ratios (FP4 = 6x, FP8 = 2x).
    pv4 (the full-FP4 PV ablation): both products at the FP4 ratio."""
    flops = FLOP_PER_PAIR * cfg.pairs
    f4 = f8 = flops / 2
    p4, p8 = 6 * peaks["bf16"], 2 * peaks["bf16"]
    t_roof = (flops / (p4 * 1e12) if pv4 else f4 / (p4 * 1e12) + f8 / (p8 * 1e12))
    peak_eff = flops / t_roof / 1e12
    achieved = flops / (pre_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak_eff, "unit": "TFLOP/s",
            "frac": achieved / peak_eff,
            "traffic": None if pv4 else measured_traffic("prefill_kernel", cfg.name),
            "traffic_unit": "bytes per launch (ncu dram read + write)",
            "algorithmic_bytes": None if pv4 else prefill_algo_bytes(cfg),
            "kernel": "prefill_kernel<true> (full-FP4 PV)" if pv4 else "prefill_kernel",
            "peak_source": peaks["source"] + (" bf16 burst x nominal FP4 ratio (6x)" if pv4 else
                                              " bf16 burst x nominal FP4 (6x) / FP8 (2x) "
                                              "ratios, harmonic mix for equal FP4 and FP8 FLOPs")}


def time_prefill(mp, cfg, Q, K, V, flush, stream, steps, warmup, compensate=True, T=T_TERMS,
                 clocks=None, k_smooth=False, pv4=False):
    """Quantize + prefill of `cfg` timed with CUDA events on the launching
    stream, L2 flushed before every step.  pv4: the full-FP4 PV ablation
    (V^T quantized to NVFP4, the FP4-PV prefill kernel) in place of the
    method's FP8 PV.  Returns (step, quantize, prefill) mean ms."""
    if pv4:
        return _time_prefill_pv4(mp, cfg, Q, K, V, flush, stream, steps, warmup, clocks)
    z = mp.quantize_qkv(Q, K, V, compensate=compensate, T=T, k_smooth=k_smooth)
    ws = z["_workspace"]
    o, lse = mp.prefill(z, causal=cfg.causal)
    for _ in range(max(warmup, 3)):
        flush.zero_()
        z = mp.quantize_qkv(Q, K, V, compensate=compensate, T=T, k_smooth=k_smooth, workspace=ws)
        mp.prefill(z, causal=cfg.causal, out=o, lse=lse)
    torch.cuda.synchronize()
    if mp.get_error() != 0:
        raise RuntimeError(f"device status word set during warm-up of {cfg.name}")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if clocks is not None:
        clocks.start()
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for ev in evs:
        flush.zero_()
        ev[0].record(stream)
        z = mp.quantize_qkv(Q, K, V, compensate=compensate, T=T, k_smooth=k_smooth, workspace=ws)
        ev[1].record(stream)
        mp.prefill(z, causal=cfg.causal, out=o, lse=lse)
        ev[2].record(stream)
    torch.cuda.synchronize()
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()
    if mp.get_error() != 0:
        raise RuntimeError(f"device status word set while timing {cfg.name}")
    return (statistics.mean(e[0].elapsed_time(e[2]) for e in evs),
            statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
            statistics.mean(e[1].elapsed_time(e[2]) for e in evs))


def _time_prefill_pv4(mp, cfg, Q, K, V, flush, stream, steps, warmup, clocks):
    z = mp.quantize_qkv(Q, K, None, compensate=True, T=T_TERMS)
    vt = mp.quantize_v_fp4(V)
    ws, wsv = z["_workspace"], vt["_workspace"]
    o, lse = mp.prefill_fp4pv(z, vt, causal=cfg.causal)

    def quant():
        return (mp.quantize_qkv(Q, K, None, compensate=True, T=T_TERMS, workspace=ws),
                mp.quantize_v_fp4(V, workspace=wsv))

    for _ in range(max(warmup, 3)):
        flush.zero_()
        zz, vv = quant()
        mp.prefill_fp4pv(zz, vv, causal=cfg.causal, out=o, lse=lse)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if clocks is not None:
        clocks.start()
    torch.cuda.synchronize()
    for ev in evs:
        flush.zero_()
        ev[0].record(stream)
        zz, vv = quant()
        ev[1].record(stream)
        mp.prefill_fp4pv(zz, vv, causal=cfg.causal, out=o, lse=lse)
        ev[2].record(stream)
    torch.cuda.synchronize()
    if mp.get_error() != 0:
        raise RuntimeError(f"device status word set while timing {cfg.name} (FP4 PV)")
    return (statistics.mean(e[0].elapsed_time(e[2]) for e in evs),
            statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
            statistics.mean(e[1].elapsed_time(e[2]) for e in evs))


def run_gpu(args):
    import flashattention_mpfa_quantize_gb300 as mp
    ws, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = _peaks()
    cfg = mi.PREFILL[args.workload]
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    launches = 0

    if args.only == "decode":
        dec = {name: run_decode(mp, dev, stream, peaks, flush, args, mi.DECODE[name])
               for name in DECODES}
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": None, "unit": "GB/s", "n_gpus": ws,
                              "steps": args.steps, "warmup": args.warmup, "decode": dec,
                              "note": "profiling aid: decode only"}), flush=True)
        return

    Q, K, V = mi.prefill_inputs(cfg, dev, seed=rank)
    clocks = Clocks(dev.index)
    pv4 = args.pv == "fp4"
    step_ms, quant_ms, pre_ms = time_prefill(mp, cfg, Q, K, V, flush, stream, args.steps,
                                             args.warmup, clocks=clocks, pv4=pv4)
    clk = clocks.stop()
    launches += (5 if pv4 else 3) * args.steps
    flops = FLOP_PER_PAIR * cfg.pairs
    rate, ms = aggregate_rate(flops, step_ms, ws, dev)
    value = rate / 1e12
    roofline = prefill_roofline(cfg, pre_ms, peaks, pv4=pv4)
    roofline.update({"workload": cfg.name, "quantize_ms": quant_ms, "prefill_ms": pre_ms})
    # diagnostic: the exp-unit bound (one ex2 per pair at 32 per clock per SM)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    f_clk = (clk or {}).get("sm_mhz") or 2070.0
    t_exp = cfg.pairs / (n_sm * 32 * f_clk * 1e6) * 1e3
    roofline["exp_unit"] = {"bound_ms": t_exp, "frac": t_exp / pre_ms, "sm_mhz": f_clk,
                            "rate": "32 ex2 per clock per SM"}

    extra = {}
    if args.only is None:
        few = max(3, min(args.steps, 5))
        roofline["compensation"] = compensation_cost(mp, cfg, Q, K, V, flush, stream, few)
        extra["bf16_sdpa"] = bf16_sdpa_baseline(Q, K, V, cfg, flush, stream, few, flops,
                                                step_ms, pre_ms)
        extra["pv_fp4_ablation"] = pv_fp4_ablation(mp, cfg, Q, K, V, flush, stream,
                                                   max(2, min(args.steps, 3)))
        e2e = run_e2e(mp, dev, stream, cfg, Q, K, V, max(3, min(args.steps, 20)))
        launches += 3 * max(3, min(args.steps, 20)) + 6
    else:
        e2e = None

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and args.only is None:
        try:
            heads = tuple((0, h) for h in range(0, cfg.Hq, max(1, cfg.Hq // 4)))[:4]
            v, dt, desc, thr = oracle_sample(cfg, Q.cpu(), K.cpu(), V.cpu(), rows_per_head=128,
                                             heads=heads)
            cpu = {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                   "sample": desc, "seconds": dt}
        except Exception as ex:  # pragma: no cover - reported, not fatal
            cpu = {"error": repr(ex)}
    del Q, K, V
    torch.cuda.empty_cache()

    other = {}
    if args.only is None and not args.no_secondary:
        for name in OTHER_PREFILL:
            if name == cfg.name:
                continue
            c2 = mi.PREFILL[name]
            q2, k2, v2 = mi.prefill_inputs(c2, dev, seed=rank)
            n2 = max(3, min(args.steps, 20))
            s2, qm2, pm2 = time_prefill(mp, c2, q2, k2, v2, flush, stream, n2, 3)
            launches += 3 * n2
            r2 = prefill_roofline(c2, pm2, peaks)
            r2.pop("peak_source")
            other[name] = {"value": FLOP_PER_PAIR * c2.pairs / (s2 * 1e-3) / 1e12,
                           "unit": "TFLOP/s", "ms_per_step": s2, "quantize_ms": qm2,
                           "prefill_ms": pm2, "roofline": r2}
            del q2, k2, v2
            torch.cuda.empty_cache()

    dec = {}
    if args.only is None:
        for name in DECODES:
            d = run_decode(mp, dev, stream, peaks, flush, args, mi.DECODE[name])
            launches += d.pop("gpu_launches")
            dec[name] = d

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": ("nvfp4 e2m1 (QK and PV: full-FP4 ablation), fp32 accumulate" if pv4
                          else "nvfp4 e2m1 (QK) + fp8 e4m3 (PV), fp32 accumulate"),
                "data": "synthetic",
                "config": {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
                           "N": cfg.N, "d": 128, "causal": cfg.causal, "compensate": True,
                           "T": T_TERMS,
                           "step": ("mpfa_quantize_qkv (Q, K) + mpfa_quantize_v_fp4 + "
                                    "mpfa_prefill_fp4pv" if pv4
                                    else "mpfa_quantize_qkv + mpfa_prefill"),
                           "l2": "inputs larger than L2, and L2 flushed (512 MB write) before "
                                 "every step",
                           "parallelism": "replicas" if ws > 1 else "single"},
                "roofline": roofline, "prefill_other": other, "decode": dec, "e2e": e2e,
                "cpu_baseline": cpu, "gpu_launches": launches, "clocks": clk, **extra}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def bf16_sdpa_baseline(Q, K, V, cfg, flush, stream, steps, flops, step_ms, pre_ms):
    """Context, not part of the product: torch's fused bf16 attention backends
    (cuDNN, flash) on the same unquantized inputs, each timed the same way;
    the ratios are against the fastest one."""
    from torch.nn.attention import SDPBackend, sdpa_kernel
    import torch.nn.functional as F
    q, k, v = (t.transpose(1, 2).contiguous() for t in (Q, K, V))   # [B, H, N, d]
    out = {}
    for name, be in (("cudnn", SDPBackend.CUDNN_ATTENTION),
                     ("flash", SDPBackend.FLASH_ATTENTION)):
        try:
            with sdpa_kernel([be]):
                def run():
                    return F.scaled_dot_product_attention(q, k, v, is_causal=cfg.causal,
                                                          enable_gqa=cfg.Hq != cfg.Hkv)
                for _ in range(2):
                    run()
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(max(steps, 1))]
                for a, b in evs:
                    flush.zero_()
                    a.record(stream)
                    run()
                    b.record(stream)
                torch.cuda.synchronize()
            out[name] = statistics.mean(a.elapsed_time(b) for a, b in evs)
        except Exception as ex:  # pragma: no cover - a backend torch lacks here
            out[name] = "unavailable: " + repr(ex)[:120]
    del q, k, v
    times = {n: t for n, t in out.items() if isinstance(t, float)}
    if not times:
        return {"unavailable": out}
    best = min(times, key=times.get)
    ms = times[best]
    return {"kernel": "torch scaled_dot_product_attention, bf16", "ms_by_backend": out,
            "fastest": best, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
            "speedup_of_step": ms / step_ms, "speedup_of_prefill_kernel": ms / pre_ms}


def compensation_cost(mp, cfg, Q, K, V, flush, stream, steps):
    """Quantize and prefill times with the rank-one compensation off, with one
    and with two terms, and with two terms plus key-side smoothing, timed in
    interleaved rounds (so clock and power drift hit every variant alike)."""
    variants = {"off": dict(compensate=False), "T1": dict(compensate=True, T=1),
                "T2": dict(compensate=True, T=2),
                "T2_ksmooth": dict(compensate=True, T=2, k_smooth=True)}
    acc = {k: ([], []) for k in variants}
    for _ in range(steps):
        for k, kw in variants.items():
            _, q, p = time_prefill(mp, cfg, Q, K, V, flush, stream, 1, 1, **kw)
            acc[k][0].append(q)
            acc[k][1].append(p)
    out = {"rounds": steps}
    for k in variants:
        out[f"quantize_ms_{k}"] = statistics.mean(acc[k][0])
        out[f"prefill_ms_{k}"] = statistics.mean(acc[k][1])
    p_off, q_off = out["prefill_ms_off"], out["quantize_ms_off"]
    for k in ("T1", "T2", "T2_ksmooth"):
        out[f"prefill_overhead_pct_{k}"] = 100.0 * (out[f"prefill_ms_{k}"] / p_off - 1.0)
        out[f"step_overhead_pct_{k}"] = 100.0 * ((out[f"quantize_ms_{k}"] + out[f"prefill_ms_{k}"])
                                                 / (q_off + p_off) - 1.0)
    return out


def pv_fp4_ablation(mp, cfg, Q, K, V, flush, stream, steps):
    """The MpFA abstract's trade-off measured: the method's FP8 PV step
    (quantize Q, K, V + prefill) against the full-FP4 PV step (quantize Q, K;
    V^T in NVFP4; the FP4-PV prefill kernel), timed in interleaved rounds with
    CUDA events, L2 flushed before each; and both outputs' rel-L2 against
    torch's bf16 attention on four query heads (context for the accuracy
    side; the parity tests check each kernel against the oracle)."""
    z8 = mp.quantize_qkv(Q, K, V, compensate=True, T=T_TERMS)
    z4 = mp.quantize_qkv(Q, K, None, compensate=True, T=T_TERMS)
    vt = mp.quantize_v_fp4(V)
    o8, l8 = mp.prefill(z8, causal=cfg.causal)
    o4, l4 = mp.prefill_fp4pv(z4, vt, causal=cfg.causal)
    ws8, ws4, wsv = z8["_workspace"], z4["_workspace"], vt["_workspace"]

    def step8():
        z = mp.quantize_qkv(Q, K, V, compensate=True, T=T_TERMS, workspace=ws8)
        mp.prefill(z, causal=cfg.causal, out=o8, lse=l8)

    def step4():
        z = mp.quantize_qkv(Q, K, None, compensate=True, T=T_TERMS, workspace=ws4)
        v4 = mp.quantize_v_fp4(V, workspace=wsv)
        mp.prefill_fp4pv(z, v4, causal=cfg.causal, out=o4, lse=l4)

    def kern8():
        mp.prefill(z8, causal=cfg.causal, out=o8, lse=l8)

    def kern4():
        mp.prefill_fp4pv(z4, vt, causal=cfg.causal, out=o4, lse=l4)

    fns = {"step_pv8": step8, "step_pv4": step4, "prefill_pv8": kern8, "prefill_pv4": kern4}
    for f in fns.values():
        for _ in range(2):
            flush.zero_()
            f()
    torch.cuda.synchronize()
    acc = {k: [] for k in fns}
    for _ in range(steps):
        for k, f in fns.items():
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            f()
            b.record(stream)
            b.synchronize()
            acc[k].append(a.elapsed_time(b))
    if mp.get_error() != 0:
        raise RuntimeError("device status word set in the PV precision ablation")
    out = {"rounds": steps}
    for k in fns:
        out[f"{k}_ms"] = statistics.mean(acc[k])
    out["prefill_ratio_pv4_over_pv8"] = out["prefill_pv4_ms"] / out["prefill_pv8_ms"]
    out["step_ratio_pv4_over_pv8"] = out["step_pv4_ms"] / out["step_pv8_ms"]
    q, k, v = (t.transpose(1, 2) for t in (Q, K, V))
    g = cfg.Hq // cfg.Hkv
    heads = list(range(0, cfg.Hq, max(1, cfg.Hq // 4)))[:4]
    num8 = num4 = den = 0.0
    for h in heads:
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[:, h:h + 1].contiguous(), k[:, h // g:h // g + 1].contiguous(),
            v[:, h // g:h // g + 1].contiguous(), is_causal=cfg.causal).float()[:, 0]
        num8 += (o8[:, :, h].float() - ref).pow(2).sum().item()
        num4 += (o4[:, :, h].float() - ref).pow(2).sum().item()
        den += ref.pow(2).sum().item()
        del ref
    out["heads"] = heads
    out["rel_l2_vs_bf16_sdpa_pv8"] = (num8 / den) ** 0.5
    out["rel_l2_vs_bf16_sdpa_pv4"] = (num4 / den) ** 0.5
    del z8, z4, vt, o8, o4, l8, l4
    torch.cuda.empty_cache()
    return out


def run_decode(mp, dev, stream, peaks, flush, args, cfg):
    if args.decode_batch:
        cfg = mi.custom_decode(args.decode_batch, cfg.Hq, cfg.Hkv, cfg.Lmax, cfg.len_lo,
                               cfg.len_hi, name=f"{cfg.name}_b{args.decode_batch}")
    q, K, V, seqlens = mi.decode_inputs(cfg, dev, seed=1)
    cache = mp.quantize_qkv(None, K, V)
    del K, V
    torch.cuda.empty_cache()
    res = mp.decode(q, cache, seqlens)
    ws_d = res["_workspace"]
    out, lse = res["o"], res["lse"]
    for _ in range(3):
        flush.zero_()
        mp.decode(q, cache, seqlens, out=out, lse=lse, workspace=ws_d)
    torch.cuda.synchronize()
    n = max(args.steps, 5)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    clocks = Clocks(dev.index)
    clocks.start()
    for i in range(n):
        flush.zero_()
        evs[i][0].record(stream)
        mp.decode(q, cache, seqlens, out=out, lse=lse, workspace=ws_d)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if mp.get_error() != 0:
        raise RuntimeError(f"device status word set while timing {cfg.name}")
    ms_local = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    tokens = int(seqlens.long().sum().item())
    nbytes = tokens * cfg.Hkv * KV_BYTES_PER_TOKEN
    gbs = nbytes / (ms_local * 1e-3) / 1e9          # this replica's kernel rate (roofline)
    job, ms = aggregate_rate(nbytes, ms_local, _dist()[0], dev)
    del cache
    torch.cuda.empty_cache()
    return {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "Lmax": cfg.Lmax,
            "lengths": [cfg.len_lo, cfg.len_hi], "cached_tokens": tokens,
            "value": job / 1e9, "unit": "GB/s", "ms": ms, "chunk": res["chunk"],
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"],
                         "traffic": (measured_traffic("split_kernel", cfg.name)
                                     if not args.decode_batch else None),
                         "traffic_unit": "bytes per launch (ncu dram read + write)",
                         "algorithmic_bytes": nbytes, "kernel": "split_kernel"},
            "gpu_launches": 4 * n, "clocks": clk}


def run_e2e(mp, dev, stream, cfg, Q, K, V, n):
    """Same step through the public API with pinned host buffers: every step
    copies its bf16 Q/K/V from the host, quantizes, runs the prefill and
    copies its O and LSE back to the host, all inside the timed region.  The
    copies run on two copy streams with two device buffer sets, so the upload
    of step i+1 and the download of step i-1 overlap the compute of step i."""
    hq = torch.empty(Q.shape, dtype=Q.dtype, pin_memory=True)
    hk = torch.empty(K.shape, dtype=K.dtype, pin_memory=True)
    hv = torch.empty(V.shape, dtype=V.dtype, pin_memory=True)
    hq.copy_(Q)
    hk.copy_(K)
    hv.copy_(V)
    B, N, Hq = cfg.B, cfg.N, cfg.Hq
    ho = [torch.empty(Q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    hl = [torch.empty(B, Hq, N, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    dq = [torch.empty_like(Q) for _ in range(2)]
    dk = [torch.empty_like(K) for _ in range(2)]
    dv = [torch.empty_like(V) for _ in range(2)]
    o = [torch.empty_like(Q) for _ in range(2)]
    lse = [torch.empty(B, Hq, N, dtype=torch.float32, device=dev) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = [ev(), ev()]      # inputs of buffer b uploaded
    in_free = [None, None]       # quantize of buffer b done (inputs consumed)
    out_ready = [ev(), ev()]     # O of buffer b computed
    out_free = [None, None]      # O of buffer b downloaded
    ws_q = [None, None]

    def step(i):
        b = i & 1
        with torch.cuda.stream(up):
            if in_free[b] is not None:
                up.wait_event(in_free[b])
            dq[b].copy_(hq, non_blocking=True)
            dk[b].copy_(hk, non_blocking=True)
            dv[b].copy_(hv, non_blocking=True)
            in_ready[b].record(up)
        stream.wait_event(in_ready[b])
        if out_free[b] is not None:
            stream.wait_event(out_free[b])
        z = mp.quantize_qkv(dq[b], dk[b], dv[b], compensate=True, T=T_TERMS, workspace=ws_q[b])
        ws_q[b] = z["_workspace"]
        e = ev()
        e.record(stream)
        in_free[b] = e
        mp.prefill(z, causal=cfg.causal, out=o[b], lse=lse[b])
        out_ready[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(out_ready[b])
            ho[b].copy_(o[b], non_blocking=True)
            hl[b].copy_(lse[b], non_blocking=True)
            f = ev()
            f.record(down)
            out_free[b] = f

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    up.wait_event(t0)
    for i in range(n):
        step(i)
    stream.wait_event(out_free[(n - 1) & 1])
    stream.wait_event(out_free[n & 1])
    t1.record(stream)
    torch.cuda.synchronize()
    wsz = _dist()[0]
    flops = FLOP_PER_PAIR * cfg.pairs
    rate, ms = aggregate_rate(flops, t0.elapsed_time(t1) / n, wsz, dev)
    h2d = (Q.numel() + K.numel() + V.numel()) * 2
    d2h = Q.numel() * 2 + B * Hq * N * 4
    return {"value": rate / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelining": "two buffer sets; H2D of step i+1 and D2H of step i-1 overlap step i"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(mi.PREFILL),
                    help="prefill workload of the timed step (default: the 128K headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other prefill workloads")
    ap.add_argument("--pv", choices=["fp8", "fp4"], default="fp8",
                    help="fp4: time the full-FP4 PV ablation kernel instead of the method's "
                         "FP8 PV (with --only prefill)")
    ap.add_argument("--only", choices=["prefill", "decode"], default=None,
                    help="profiling aid: time only this part (no e2e / cpu baseline)")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="profiling aid: smaller decode batch than the workload's 64")
    args = ap.parse_args()
    if args.pv == "fp4" and args.only != "prefill":
        ap.error("--pv fp4 times the ablation kernel alone: give --only prefill")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

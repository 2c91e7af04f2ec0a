"""Benchmark: CSA prefill of 1 x 8192 tokens on one B300 (tokens/s).

One step = the whole CSA hot path over one batch of synthetic input, through
the C ABI of libcsa_b300.so: block compression of the KV cache (m = 4, mixed
FP8/BF16 rows) and of the window cache (m = 1), compression of the FP4
indexer keys, lightning-indexer scores + top-k (k = 512), and sparse MQA over
the selected entries plus the 128-token window (64 heads, D = 512).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With torchrun (N > 1) every rank runs its own sequence (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
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

import workloads as wl  # noqa: E402

CFG = wl.CONFIGS["c2_csa_prefill_8k"]
METRIC = "CSA prefill tokens/s (1x8192, m=4, top-k 512, window 128, 64 heads, D=512)"


def attn_flops(cfg) -> float:
    """Algorithmic flops of the sparse MQA step: per query and head 4D per key
    (QK^T and PV), keys = min(k, visible entries) + min(W, t + 1)."""
    t = np.arange(cfg.T, dtype=np.int64)
    keys = np.minimum(cfg.k, np.minimum(cfg.N, (t + 1) // cfg.m)) + np.minimum(cfg.W, t + 1)
    return float(keys.sum()) * cfg.H * 4 * cfg.D


def indexer_flops(cfg) -> float:
    t = np.arange(cfg.T, dtype=np.int64)
    pairs = np.minimum(cfg.N, (t + 1) // cfg.m).sum()
    return float(pairs) * 2 * cfg.HI * cfg.dI


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thr = threading.Thread(target=self._read, daemon=True)
            self.thr.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        sm = [float(r[0]) for r in self.rows if len(r) >= 7 and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) >= 7 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) >= 7 for i in range(4)
                          if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm)}


# --------------------------------------------------------------------------
# ranks (torchrun, N > 1): each rank runs its own sequence; the times are
# reduced by max, the value counts every rank's tokens
# --------------------------------------------------------------------------
def max_over_ranks(values, dist, device):
    """The per-rank times, each replaced by its maximum over the ranks."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def aggregate_tokens_per_s(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Whole-job throughput: all ranks' tokens over the slowest rank's step."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


# --------------------------------------------------------------------------
# inputs
# --------------------------------------------------------------------------
def host_inputs(seed: int):
    toks = wl.gen_tokens(CFG, 0, seed=seed)
    qry = wl.gen_queries(CFG, 0, seed=seed)
    sc = wl.gen_channel_scales(CFG, seed=seed)
    return {"kv": toks["kv"][None], "z": toks["z"][None], "kI": toks["kI"][None], "zI": toks["zI"][None],
            "q": qry["q"][None], "qI": qry["qI"][None], "w": qry["w"][None], "s": sc["s"], "sI": sc["sI"],
            "q_pos": np.arange(CFG.T, dtype=np.int64)[None], "swa_pos0": np.zeros(1, np.int64)}


BF16_KEYS = ("kv", "kI", "q", "qI")


def bench_config(world: int) -> dict:
    """The workload description both arms print (identical dicts)."""
    return {"workload": CFG.name, "B": 1, "T": CFG.T, "m": CFG.m, "N": CFG.N, "k": CFG.k, "W": CFG.W,
            "H": CFG.H, "D": CFG.D, "HI": CFG.HI, "dI": CFG.dI, "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (q and out 512 MiB each per step)"}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    import torch
    import long_context_sparse_29_b300 as csa
    from long_context_sparse_29_b300 import build as csa_build

    csa_build.build()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    h = host_inputs(seed=rank)
    pinned = {}
    for kname, a in h.items():
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if kname in BF16_KEYS else a)
        if kname in BF16_KEYS:
            t = t.view(torch.bfloat16)
        pinned[kname] = t.pin_memory()
    d = {kname: t.cuda() for kname, t in pinned.items()}
    rope = csa.rope_table(CFG.T + 1, CFG.R)
    scale = 1.0 / math.sqrt(CFG.D)
    T, N, m, k, W = CFG.T, CFG.N, CFG.m, CFG.k, CFG.W
    dev = torch.device("cuda", local_rank)
    cache = torch.empty((1, N, 592), dtype=torch.uint8, device=dev)
    swa = torch.empty((1, T, 592), dtype=torch.uint8, device=dev)
    kcodes = torch.empty((1, N, CFG.dI // 2), dtype=torch.uint8, device=dev)
    kscales = torch.empty((1, N, CFG.dI // 32), dtype=torch.uint8, device=dev)
    idx = torch.empty((1, T, k), dtype=torch.int32, device=dev)
    out = torch.empty((1, T, CFG.H, CFG.D), dtype=torch.bfloat16, device=dev)
    ws = csa.Workspace(dev)
    stream = torch.cuda.current_stream(dev)
    ev_attn = []

    def step(x, timed=False):
        csa.compress_kv(x["kv"], x["z"], x["s"], m, csa.FMT_MIXED592, CFG.R, rope, out=cache)
        csa.compress_kv(x["kv"], x["z"], None, 1, csa.FMT_MIXED592, CFG.R, rope, out=swa)
        csa.compress_kv(x["kI"], x["zI"], x["sI"], m, csa.FMT_MXFP4, 0, out=kcodes, out_scales=kscales)
        csa.indexer_topk(x["qI"], x["w"], kcodes, kscales, x["q_pos"], N, m, k, scores=False,
                         idx_out=idx, ws=ws)
        if timed:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        csa.sparse_mqa(x["q"], x["q_pos"], cache, m, idx, swa, x["swa_pos0"], W, scale, rope,
                       CFG.R, out=out, ws=ws)
        if timed:
            e1.record(stream)
            ev_attn.append((e0, e1))

    for _ in range(args.warmup):
        step(d)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step(d, timed=True)
        t1.record(stream)
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_attn)
    flags = ws.flags()
    if flags:
        raise RuntimeError(f"device check flags {flags} during the benchmark")

    # end to end through the public API with host buffers: H2D of the step's inputs,
    # the step, D2H of the output
    in_keys = ("kv", "z", "kI", "zI", "q", "qI", "w", "s", "sI", "q_pos", "swa_pos0")
    h2d = sum(pinned[kname].numel() * pinned[kname].element_size() for kname in in_keys)
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(2, min(args.steps, 5))
    dd = {kname: torch.empty_like(d[kname]) for kname in in_keys}

    def e2e_step():
        for kname in in_keys:
            dd[kname].copy_(pinned[kname], non_blocking=True)
        step(dd)
        host_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    if dist:
        ms, e2e_ms, attn_ms = max_over_ranks([ms, e2e_ms, attn_ms], dist, dev)
    pk = peaks()
    af = attn_flops(CFG)
    achieved = af / (attn_ms * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    fp8_peak = 2.0 * peak   # dense FP8 = the measured bf16 burst x the nominal 2x ratio
    ms_step = ms / args.steps
    step_flops = af + indexer_flops(CFG)
    res = {
        "metric": METRIC, "value": aggregate_tokens_per_s(world, T, ms_step), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world),
        "roofline": {"kernel": "sparse_mqa", "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": ATTN_TRAFFIC,
                     "peak_src": f"bf16 dense, {pk['src']} (burst)",
                     "algorithmic_flops_per_launch": af, "avg_launch_ms": attn_ms},
        # the same attention launch against the dense FP8 tensor roofline, and the
        # whole step (indexer + attention flops over the step time) against it
        "roofline_fp8": {"kernel": "sparse_mqa", "bound": "tensor", "achieved": achieved, "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                         "peak_src": f"dense FP8 = 2 x bf16 dense, {pk['src']} (burst)"},
        "step_frac_fp8": step_flops / (ms_step * 1e-3) / 1e12 / fp8_peak,
        "step_flops": step_flops,
        "e2e": {"value": aggregate_tokens_per_s(world, T, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_decode:
        # the 1M-context decode target, measured in the same run: the hybrid
        # CSA + HCA layer pair, 4 sequences, one CUDA graph per step
        dec = run_config(argparse.Namespace(steps=max(args.steps, 20), warmup=max(args.warmup, 3)),
                         "c5_hybrid_csa_decode_1m")
        r = dec["roofline"]
        res["decode_1m"] = {"workload": dec["config"]["workload"], "metric": dec["metric"], "value": dec["value"],
                            "unit": dec["unit"], "ms_per_step": dec["ms_per_step"], "steps": dec["steps"],
                            "algorithmic_bytes_per_step": r["algorithmic_bytes_per_step"],
                            "achieved_gbs": r["achieved"], "peak_gbs": r["peak"], "hbm_frac": r["frac"],
                            "traffic_per_step": r["traffic"],
                            "peak_src": r["peak_src"], "gpu_launches": dec["gpu_launches"],
                            "clocks": dec["clocks"], "step": dec["config"]["step"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(h)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return res


# kernels launched per step: 3 compress; the indexer's query quantisation,
# entry expansion, tensor-core scores and top-k; for the attention the per-row
# prep (rotated query dims, entry lists), the bf16 expansion of the cache and
# of the window rows, and the attention kernel
LAUNCHES_PER_STEP = 11

# DRAM bytes (read + write) of one attn_tc_kernel launch on this workload, from
# one ncu capture of it (dram__bytes_read.sum + dram__bytes_write.sum); to be
# set to None when the kernel changes, until it is captured again
ATTN_TRAFFIC = 631751936 + 493387520

# DRAM bytes (read + write) of one decode step of the 4 x 1M hybrid workload:
# the sum over the step's six kernels (CSA append, scores, top-k, attention;
# HCA append, attention), from ncu captures of the current kernels (cold cache:
# dram__bytes_read.sum + dram__bytes_write.sum; nothing is written back
# within a launch); None where no capture covers every kernel of the step
DECODE_STEP_TRAFFIC = {"c5_hybrid_csa_decode_1m": 69888 + 35717120 + 4297728 + 3613696 + 575488 + 20105216}


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------
def oracle_sample(h, rows, rope):
    """One bounded oracle step: compression of all tokens, then top-k and
    attention for the given query rows.  Returns (compress s, rows s)."""
    import oracle
    t0 = time.perf_counter()
    x = wl.bf16_bits_to_f32(h["kv"])
    cache = oracle.compress_kv(x, h["z"], h["s"], CFG.m, "mixed592", CFG.R, 0, rope)
    swa = oracle.compress_kv(x, h["z"], None, 1, "mixed592", CFG.R, 0, rope)
    keys = oracle.compress_kv(wl.bf16_bits_to_f32(h["kI"]), h["zI"], h["sI"], CFG.m, "mxfp4", 0)
    t1 = time.perf_counter()
    # only the sampled rows' queries are widened to fp32
    idx, _ = oracle.indexer_topk(wl.bf16_bits_to_f32(h["qI"][:, rows]), h["w"][:, rows], keys,
                                 h["q_pos"][:, rows], CFG.N, CFG.m, CFG.k)
    oracle.attention(wl.bf16_bits_to_f32(h["q"][:, rows]), h["q_pos"][:, rows], cache, CFG.N, CFG.m,
                     idx, swa, h["swa_pos0"], CFG.W, 1.0 / math.sqrt(CFG.D), rope, CFG.R)
    return t1 - t0, time.perf_counter() - t1


def _full_step_seconds(t_comp, t_rows, n_rows):
    """Estimated oracle time of a whole 8192-token step from a sampled one."""
    return t_comp + t_rows * CFG.T / n_rows


def host_cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo; "unknown" elsewhere)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


ORACLE_ROWS = 256   # query rows per sampled oracle step (both CPU arms)


def oracle_step_seconds(h, rope, rng, n_rows=ORACLE_ROWS):
    """One sampled oracle step, scaled to the whole 8192-token step (seconds)."""
    rows = np.sort(rng.choice(CFG.T, n_rows, replace=False))
    tc, tr = oracle_sample(h, rows, rope)
    return _full_step_seconds(tc, tr, n_rows)


def oracle_sample_desc(n_rows: int) -> str:
    return (f"per step: compression of all {CFG.T} tokens + top-k and sparse MQA for {n_rows} seeded "
            f"query rows, row time scaled to {CFG.T} rows")


def cpu_baseline(h, steps=3):
    """The oracle on the host cores: the mean of `steps` sampled steps (the
    same sample as the reference arm's steps), as tokens/s."""
    import oracle
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    rope = oracle.rope_table(CFG.T + 1, CFG.R)
    rng = np.random.default_rng(123)
    secs = statistics.mean(oracle_step_seconds(h, rope, rng) for _ in range(steps))
    return {"value": CFG.T / secs, "unit": "tokens/s", "cores": oracle.get_threads(), "kind": "oracle",
            "cpu": host_cpu_model(), "rows_sampled": ORACLE_ROWS, "steps": steps,
            "sample": oracle_sample_desc(ORACLE_ROWS)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    h = host_inputs(seed=0)
    import oracle
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    rope = oracle.rope_table(CFG.T + 1, CFG.R)
    rng = np.random.default_rng(7)
    fulls = []
    for i in range(args.warmup + args.steps):
        s = oracle_step_seconds(h, rope, rng)
        if i >= args.warmup:
            fulls.append(s)
    ms = 1e3 * statistics.mean(fulls)
    value = CFG.T / (ms * 1e-3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.get_threads(), "kind": "oracle",
                         "cpu": host_cpu_model(), "rows_sampled": ORACLE_ROWS,
                         "sample": oracle_sample_desc(ORACLE_ROWS)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# --------------------------------------------------------------------------
# the other configurations (--config): decode steps against resident caches,
# and the 64K HCA prefill
# --------------------------------------------------------------------------
def _bf16_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _f_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def decode_layer(csa, cfg, dev, rope):
    """Resident decode state of one layer (every sequence's full context run
    through the library's compression into a LayerCache: entries, indexer
    keys, the last W tokens in a 2W-row window buffer, the ring of the last m
    raw tokens) and the step's inputs on the host: the query of position T-1
    and that token's activations, which the step appends again (closing block
    N-1, so every step does the append's full work and leaves the same bytes)."""
    import torch
    B, T, W, N, m = cfg.B, cfg.T, cfg.W, cfg.N, cfg.m
    sc = wl.gen_channel_scales(cfg)
    CI = cfg.dI if cfg.k else 0
    lc = csa.LayerCache(B, N, m, W, 2 * W, CI=CI, C=cfg.D, pos0=T - W, device=dev)
    new = {"kv": [], "z": [], "kI": [], "zI": []}
    for b in range(B):
        toks = wl.gen_tokens(cfg, b, parts=("kv", "z", "kI", "zI") if cfg.k else ("kv", "z"))
        kv, z = _bf16_dev(toks["kv"], dev)[None], _f_dev(toks["z"], dev)[None]
        csa.compress_kv(kv, z, _f_dev(sc["s"], dev), m, csa.FMT_MIXED592, cfg.R, rope, out=lc.cache[b:b + 1])
        csa.compress_kv(kv[:, T - W:], z[:, T - W:], None, 1, csa.FMT_MIXED592, cfg.R, rope, pos0=T - W,
                        out=lc.swa[b:b + 1, :W])
        lc.kv_tail[b] = kv[0, T - m:]
        lc.z_tail[b] = z[0, T - m:]
        if cfg.k:
            kI, zI = _bf16_dev(toks["kI"], dev)[None], _f_dev(toks["zI"], dev)[None]
            csa.compress_kv(kI, zI, _f_dev(sc["sI"], dev), m, csa.FMT_MXFP4, 0, out=lc.kI_codes[b:b + 1],
                            out_scales=lc.kI_scales[b:b + 1])
            lc.kI_tail[b] = kI[0, T - m:]
            lc.zI_tail[b] = zI[0, T - m:]
        for kk in new:
            if kk in toks:
                new[kk].append(toks[kk][T - 1])
        del kv, z, toks
    qry = [wl.gen_queries(cfg, b) for b in range(B)]
    host = {"q": np.stack([x["q"] for x in qry]), "q_pos": np.full((B, 1), T - 1, np.int64),
            "t_pos": np.full(B, T - 1, np.int64), "s": sc["s"],
            "kv_new": np.stack(new["kv"]), "z_new": np.array(new["z"], np.float32)}
    if cfg.k:
        host["qI"] = np.stack([x["qI"] for x in qry])
        host["w"] = np.stack([x["w"] for x in qry])
        host["kI_new"] = np.stack(new["kI"])
        host["zI_new"] = np.array(new["zI"], np.float32)
        host["sI"] = sc["sI"]
    return lc, host


def decode_bytes(cfg) -> float:
    """Algorithmic HBM bytes of one decode step: every resident byte the step
    must read once (indexer keys 34 B per entry; the k + W gathered or all
    visible rows, 592 B each) plus the query and the output (64 KiB each),
    and the append: the new token in, the m ring rows read, one window row and
    one entry (+ its 34-byte key) written."""
    rows = (cfg.k if cfg.k else cfg.N) + cfg.W
    per_q = rows * 592 + 2 * cfg.H * cfg.D * 2 + (cfg.N * 34 if cfg.k else 0)
    append = (cfg.m + 1) * (2 * cfg.D + 4) + 2 * 592 + ((cfg.m + 1) * (2 * cfg.dI + 4) + 34 if cfg.k else 0)
    return float(cfg.B * (per_q + append))


def decode_layer_kernels(cfg, sms):
    """Kernels one decode layer launches per step, by the library's rule: a
    row's 64-key tiles are split over min(SMs // rows, tiles) items (for at
    most 8 items the device must also hold every row's cluster at once, true
    for these configurations); items of at most 4 tiles expand the cache rows
    themselves, longer ones read rows gathered by one more kernel."""
    tiles = -(-((cfg.k if cfg.k else cfg.N) + cfg.W) // 64)
    splits = max(1, min(sms // cfg.B, tiles))
    gather = -(-tiles // splits) > 4
    return 1 + (2 if cfg.k else 0) + 1 + (1 if gather else 0)


def run_config(args, name):
    import torch
    import long_context_sparse_29_b300 as csa
    from long_context_sparse_29_b300 import build as csa_build

    csa_build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    stream = torch.cuda.current_stream(dev)
    if name in ("c3_csa_decode_128k", "c4_hca_decode_1m", "c5_hybrid_csa_decode_1m"):
        layers = [wl.CONFIGS[name]]
        if name == "c5_hybrid_csa_decode_1m":
            layers.append(wl.CONFIGS["c5_hybrid_hca_decode_1m"])
        rope = csa.rope_table(layers[0].T + 1, 64)
        built = []
        for cfg in layers:
            lc, host = decode_layer(csa, cfg, dev, rope)
            d = {kk: (_bf16_dev(v, dev) if kk in ("q", "qI", "kv_new", "kI_new") else _f_dev(v, dev))
                 for kk, v in host.items()}
            out = torch.empty((cfg.B, 1, cfg.H, cfg.D), dtype=torch.bfloat16, device=dev)
            idx = torch.empty((cfg.B, 1, cfg.k), dtype=torch.int32, device=dev) if cfg.k else None
            built.append((cfg, lc, d, out, idx, csa.Workspace(dev), csa.Workspace(dev)))
        torch.cuda.synchronize()

        def step():
            for cfg, lc, d, out, idx, ws1, ws2 in built:
                scale = 1.0 / math.sqrt(cfg.D)
                csa.decode_append(lc, d["kv_new"], d["z_new"], d["t_pos"], rope, d.get("kI_new"), d.get("zI_new"),
                                  d["s"], d.get("sI"), cfg.R)
                if cfg.k:
                    csa.indexer_topk(d["qI"], d["w"], lc.kI_codes, lc.kI_scales, d["q_pos"], cfg.N, cfg.m, cfg.k,
                                     scores=False, idx_out=idx, ws=ws1)
                    csa.sparse_mqa(d["q"], d["q_pos"], lc.cache, cfg.m, idx, lc.swa, lc.swa_pos0, cfg.W,
                                   scale, rope, cfg.R, out=out, ws=ws2)
                else:
                    csa.hca_dense_attn(d["q"], d["q_pos"], lc.cache, cfg.m, lc.swa, lc.swa_pos0, cfg.W,
                                       scale, rope, cfg.R, out=out, ws=ws2)

        graph = True
        units, unit = float(layers[0].B), "queries/s"
        metric = {"c3_csa_decode_128k": "CSA decode queries/s (32 sequences at 128K context, top-k 1024)",
                  "c4_hca_decode_1m": "HCA decode queries/s (16 sequences at 1M context, m'=128)",
                  "c5_hybrid_csa_decode_1m": "hybrid CSA+HCA decode queries/s (4 sequences at 1M, one CSA and one HCA "
                                              "layer per query)"}[name]
        alg = sum(decode_bytes(c) for c in layers)
        roof = {"bound": "hbm", "peak": pk["hbm_gbs"], "unit": "GB/s", "algorithmic_bytes_per_step": alg}
        l2 = "caches resident; each step reads them once (larger than L2 except the HCA-only step)"
        step_desc = "decode_append + indexer_topk + sparse_mqa (CSA) / decode_append + hca_dense_attn (HCA), " \
                    "one CUDA graph per step"
        # kernels per step: per layer the append; for CSA the scores (with
        # the score histogram) and the histogram top-k; the attention, and
        # before it the row gather when the attention's items are long
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        launches = sum(decode_layer_kernels(c, sms) for c in layers)
    elif name == "c2_csa_prefill_128k":
        cfg = wl.CONFIGS[name]
        T, W, m, Tc = cfg.T, cfg.W, cfg.m, 8192
        rope = csa.rope_table(T + 1, 64)
        sc = wl.gen_channel_scales(cfg)
        s_d, sI_d = _f_dev(sc["s"], dev), _f_dev(sc["sI"], dev)
        kv = torch.empty((1, T, cfg.D), dtype=torch.bfloat16, device=dev)
        kI = torch.empty((1, T, cfg.dI), dtype=torch.bfloat16, device=dev)
        z = torch.empty((1, T), dtype=torch.float32, device=dev)
        zI = torch.empty((1, T), dtype=torch.float32, device=dev)
        q = torch.empty((1, T, cfg.H, cfg.D), dtype=torch.bfloat16, device=dev)
        qI = torch.empty((1, T, cfg.HI, cfg.dI), dtype=torch.bfloat16, device=dev)
        w = torch.empty((1, T, cfg.HI), dtype=torch.float32, device=dev)
        for t0 in range(0, T, Tc):   # seeded inputs, generated chunk by chunk
            toks = wl.gen_tokens(cfg, 0, t0, t0 + Tc)
            qry = wl.gen_queries(cfg, 0, t0, t0 + Tc)
            kv[0, t0:t0 + Tc] = _bf16_dev(toks["kv"], dev)
            kI[0, t0:t0 + Tc] = _bf16_dev(toks["kI"], dev)
            z[0, t0:t0 + Tc] = _f_dev(toks["z"], dev)
            zI[0, t0:t0 + Tc] = _f_dev(toks["zI"], dev)
            q[0, t0:t0 + Tc] = _bf16_dev(qry["q"], dev)
            qI[0, t0:t0 + Tc] = _bf16_dev(qry["qI"], dev)
            w[0, t0:t0 + Tc] = _f_dev(qry["w"], dev)
            del toks, qry
        out = torch.empty_like(q)
        cp = csa.ChunkedPrefill(T, m, cfg.k, W, rope, device=dev)
        scale = 1.0 / math.sqrt(cfg.D)

        def step():
            for t0 in range(0, T, Tc):
                t1 = t0 + Tc
                cp.run(t0, t1, kv[:, t0:t1], z[:, t0:t1], kI[:, t0:t1], zI[:, t0:t1], s_d, sI_d, q[:, t0:t1],
                       qI[:, t0:t1], w[:, t0:t1], scale, out=out[:, t0:t1])

        units, unit = float(T), "tokens/s"
        metric = "CSA prefill tokens/s (1x131072 in chunks of 8192, m=4, top-k 512, window 128, 64 heads, D=512)"
        t = np.arange(T, dtype=np.int64)
        keys = np.minimum(cfg.k, (t + 1) // m) + np.minimum(W, t + 1)
        alg = float(keys.sum()) * cfg.H * 4 * cfg.D
        roof = {"bound": "tensor", "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "algorithmic_flops_per_step": alg}
        l2 = "inputs larger than L2 (q and out 8 GiB each)"
        layers = [cfg]
        graph = False
        step_desc = ("16 chunks of 8192 tokens, each: compress (entries, window rows, keys) + indexer_topk + "
                     "sparse_mqa against the caches so far; roofline = attention flops over the whole step")
        launches = 16 * LAUNCHES_PER_STEP   # the 8K step's 11 kernels per chunk
    elif name == "c4_hca_prefill_64k":
        cfg = wl.CONFIGS[name]
        T, W, N, m = cfg.T, cfg.W, cfg.N, cfg.m
        rope = csa.rope_table(T + 1, 64)
        sc = wl.gen_channel_scales(cfg)
        toks = wl.gen_tokens(cfg, 0, parts=("kv", "z"))
        qry = wl.gen_queries(cfg, 0)
        kv, z = _bf16_dev(toks["kv"], dev)[None], _f_dev(toks["z"], dev)[None]
        q = _bf16_dev(qry["q"], dev)[None]
        q_pos = _f_dev(np.arange(T, dtype=np.int64)[None], dev)
        pos0 = _f_dev(np.zeros(1, np.int64), dev)
        s_d = _f_dev(sc["s"], dev)
        cache = torch.empty((1, N, 592), dtype=torch.uint8, device=dev)
        swa = torch.empty((1, T, 592), dtype=torch.uint8, device=dev)
        out = torch.empty((1, T, cfg.H, cfg.D), dtype=torch.bfloat16, device=dev)
        ws = csa.Workspace(dev)
        scale = 1.0 / math.sqrt(cfg.D)

        def step():
            csa.compress_kv(kv, z, s_d, m, csa.FMT_MIXED592, cfg.R, rope, out=cache)
            csa.compress_kv(kv, z, None, 1, csa.FMT_MIXED592, cfg.R, rope, out=swa)
            csa.hca_dense_attn(q, q_pos, cache, m, swa, pos0, W, scale, rope, cfg.R, out=out, ws=ws)

        units, unit = float(T), "tokens/s"
        metric = "HCA prefill tokens/s (1x65536, m'=128, window 128, 64 heads, D=512)"
        t = np.arange(T, dtype=np.int64)
        keys = np.minimum(N, (t + 1) // m) + np.minimum(W, t + 1)
        alg = float(keys.sum()) * cfg.H * 4 * cfg.D
        roof = {"bound": "tensor", "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "algorithmic_flops_per_step": alg}
        l2 = "inputs larger than L2 (q and out 4 GiB each)"
        layers = [cfg]
        graph = False
        step_desc = "compress (entries and window rows) + hca_dense_attn"
        launches = 6   # 2 compress; row prep, cache and window expansion, attention
    else:
        raise SystemExit(f"unknown config {name}")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    run = step
    if graph:
        # the step's launches captured once (workspaces already sized by the
        # warm-up steps) and replayed: no host work between kernels
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        run = g.replay
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            run()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    if roof["bound"] == "hbm":
        ach = roof["algorithmic_bytes_per_step"] / (ms * 1e-3) / 1e9
    else:
        ach = roof["algorithmic_flops_per_step"] / (ms * 1e-3) / 1e12
    roof.update({"achieved": ach, "frac": ach / roof["peak"], "traffic": DECODE_STEP_TRAFFIC.get(name),
                 "peak_src": f"{pk['src']} ({'HBM copy' if roof['bound'] == 'hbm' else 'bf16 dense, burst'})",
                 "note": "the whole step (all its launches) timed with CUDA events"})
    cfg0 = layers[0]
    return {"metric": metric, "value": units / (ms * 1e-3), "unit": unit, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": name, "B": cfg0.B, "T": cfg0.T, "N": cfg0.N, "m": cfg0.m, "k": cfg0.k,
                       "W": cfg0.W, "H": cfg0.H, "D": cfg0.D, "l2": l2, "step": step_desc},
            "roofline": roof, "gpu_launches": launches * args.steps, "clocks": clk.summary()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the 1M-context decode measurement")
    ap.add_argument("--config", default=CFG.name,
                    help="workload; the default is the 8K CSA prefill, the others are measured on one GPU")
    args = ap.parse_args()
    if args.config != CFG.name:
        if args.impl != "ours":
            raise SystemExit("--config applies to --impl ours only")
        print(json.dumps(run_config(args, args.config)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

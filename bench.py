"""Benchmark of the KDA hot path on GB300: chunkwise prefill (headline) plus fused decode.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step = one ``kda_prefill`` call over the prefill workload (B=1, H=96,
T=8192, dk=dv=128, bf16 q/k/v, fp32 g/beta/state, N(0,0.02) initial state,
fp32 output): every stage of the chunkwise path.  The decode workload (B=256,
H=96, dk=dv=128, 64 consecutive in-place steps) is timed in the same run and
reported in the ``decode`` object, and K = 4 tokens per sequence through one
``kda_decode_multi`` call in the ``decode_multi`` object.  Inputs are larger than L2 (1.41 GB prefill,
1.61 GB decode state), so no flush is needed between iterations.  ``e2e`` times
``kda_prefill_host`` from pinned host inputs to pinned host outputs (out and final
state) every step.  ``prologue`` times the same prefill from the recipe's raw draws with the
input prologue in the kernels, ``gate`` the same prefill through ``kda_prefill_gated`` (the
output gate o * sigmoid(z)), ``checkpoints`` through ``kda_prefill_checkpointed`` (a state
snapshot every 512 tokens), ``fp32`` the same workload with fp32 q/k/v on the CUDA-core
kernel (at most 10 calls), and ``context_parallel`` the same sequence as two token ranges
emulated on this GPU (local passes, one fold, the rerun).  nvidia-smi clock samples are kept for the timed windows of
every leg.

Rank 0 prints one JSON line.  Under torchrun each rank runs its own independent
copy of the workload (weak scaling, no collective on the data path).
``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import kda_workloads as W  # noqa: E402

METRIC = "KDA prefill tokens/s (×tensor-peak %) and decode state GB/s (×HBM-peak %), 1 GB300"
UNIT = "tokens/s"
E2E_SEGMENT_TOKENS = 1024
# GB300's nominal HBM3e bandwidth.  The roofline's `peak` is the measured copy bandwidth (a
# plain copy reaches less than a read-modify-write stream does, so a kernel can pass it); each
# roofline object also carries its fraction of this nominal figure.
NOMINAL_HBM_GBS = 7900.0
# the kernels one bench-size kda_prefill call runs (the chunk-parallel split path)
PREFILL_KERNEL_SRC = ("linear_attention_serving_chunkwise_gb300/csrc/kda_prefill_split.cu",
                      "linear_attention_serving_chunkwise_gb300/csrc/kda_prefill_tc_phases.cuh",
                      "linear_attention_serving_chunkwise_gb300/csrc/kda_sm100.cuh")
PREFILL_KERNELS = {1: "kda_prefill_tc_kernel",
                   2: "kda_chunk_offsets_kernel + kda_prep_scan_kernel (cooperative: chunk prep, then the state scan)",
                   3: "kda_chunk_offsets_kernel + kda_chunk_prep_kernel + kda_state_scan_kernel"}



# --------------------------------------------------------------------------- helpers
def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def prefill_algorithmic(cfg: W.PrefillConfig):
    """Algorithmic bytes and flops of one prefill call: inputs read once, output and
    final state written once; flops of the chunkwise form with 64-token chunks."""
    th = cfg.total_tokens * cfg.num_heads
    e = 2 if cfg.qkv_dtype == torch.bfloat16 else 4
    dk, dv, C = cfg.dk, cfg.dv, 64
    per_th_bytes = e * (2 * dk + dv) + 4 * dk + 4 + 4 * dv
    state_bytes = cfg.num_seqs * cfg.num_heads * dk * dv * 4 * (2 if cfg.init_state != "zero" else 1)
    per_th_flops = (C - 1) * dk + (C + 1) * dk + (C + 1) * dv + (C + 1) * dk + (C + 1) * dv + 3 * 2 * dk * dv
    return th * per_th_bytes + state_bytes, th * per_th_flops


def decode_algorithmic(cfg: W.DecodeConfig):
    """Bytes per decode step: state read + write, plus the per-token vectors and output."""
    bh = cfg.batch * cfg.num_heads
    e = 2 if cfg.qkv_dtype == torch.bfloat16 else 4
    state = bh * cfg.dk * cfg.dv * 4 * 2
    small = bh * (e * (2 * cfg.dk + cfg.dv) + 4 * cfg.dk + 4 + 4 * cfg.dv)
    return state, state + small


def _link_floor(h2d: int, d2h: int, dev) -> dict:
    """The host-device link as this box gives it: pinned 256 MB copies host-to-device,
    device-to-host and both at once (two streams), CUDA events, best of 5; and the floor
    they set for an e2e step of h2d bytes up and d2h bytes down, max(up alone, both
    directions at the combined rate).  The e2e number is read against this floor."""
    n = 256 << 20
    hbuf = [torch.empty(n, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    dbuf = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(2)]
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()

    def best(fn):
        ts = []
        for _ in range(5):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
        return min(ts)

    def up():
        with torch.cuda.stream(s0):
            dbuf[0].copy_(hbuf[0], non_blocking=True)

    def down():
        with torch.cuda.stream(s1):
            hbuf[1].copy_(dbuf[1], non_blocking=True)

    def both():
        up()
        down()

    t_up, t_down, t_both = best(up), best(down), best(both)
    h2d_gbs, d2h_gbs, both_gbs = n / t_up / 1e9, n / t_down / 1e9, 2 * n / t_both / 1e9
    floor_ms = max(h2d / (h2d_gbs * 1e9), (h2d + d2h) / (both_gbs * 1e9)) * 1e3
    del hbuf, dbuf
    return {"h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs, "both_directions_gbs": both_gbs, "floor_ms": floor_ms,
            "how": "pinned 256 MB copies, best of 5 (host wall clock around synchronised copies); floor = "
                   "max(bytes up / up rate, all bytes / both-directions rate)"}


def _src_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_tensor_pipe(src_hash: str):
    """Tensor-pipe activity of the chunk prep (sm__pipe_tensor_cycles_active, percent of the
    kernel's cycles) recorded by an ncu capture under profiles/, if taken on the current
    kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "kda_prefill_tensor_pipe.txt")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m_hash or m_hash.group(1) != src_hash:
        return None
    out = {}
    for key in ("prep_pct", "scan_pct", "prep_scan_pct"):
        m = re.search(key + r":\s*([0-9.]+)", txt)
        if m:
            out[key] = float(m.group(1))
    return out or None


def _profiled_traffic(kernel_tag: str, src_hash: str):
    """dram bytes per launch recorded by an ncu capture under profiles/, if the
    capture was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_traffic.txt")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_bytes or m_hash.group(1) != src_hash:
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 20 ms, each with its timestamp) from before the
    first timed leg to after the last.  Each timed leg marks its window (host wall clock from
    the synchronize before its first event to the synchronize after its last), and only the
    samples inside a window count: between legs the GPU idles while the host sets up."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.windows = []   # (leg, t0, t1), host wall clock
        self.path = os.path.join(tempfile.gettempdir(), f"kda_clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def window(self, leg: str, t0: float, t1: float):
        self.windows.append((leg, t0, t1))

    @staticmethod
    def _stamp(txt: str):
        import datetime
        try:
            return datetime.datetime.strptime(txt.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, per_leg, total = [], [], set(), {}, 0
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            total += 1
            ts = self._stamp(f[0])
            legs = [w[0] for w in self.windows if ts is not None and w[1] <= ts <= w[2]]
            if not legs:
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            per_leg[legs[0]] = per_leg.get(legs[0], 0) + 1
            for n, v in zip(self.NAMES, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "sm_mhz_min": min(sm) if sm else None, "reasons": sorted(reasons), "samples": len(sm),
                "samples_per_leg": per_leg, "samples_total": total, "interval_ms": 20,
                "legs": [w[0] for w in self.windows]}


# --------------------------------------------------------------------------- distributed plumbing
def _dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- CPU oracle legs
def oracle_sample(cfg: W.PrefillConfig, heads: int, tokens: int, seed: int = 0):
    """Time the oracle, as it stands, on all host cores over a bounded sample of the prefill
    workload (``heads`` heads x ``tokens`` tokens).  Returns (tokens/s scaled to all H heads,
    seconds, cores, description)."""
    import oracle
    sub = W.PrefillConfig("sample", (tokens,), heads, cfg.dk, cfg.dv, cfg.qkv_dtype, cfg.init_state)
    d = W.make_prefill_inputs(sub, seed=seed)
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"], threads=cores)
    dt = time.perf_counter() - t0
    rate = tokens * heads / dt / cfg.num_heads
    desc = (f"{heads} of {cfg.num_heads} heads x {tokens} tokens of the {cfg.name} workload, fp64 oracle, "
            f"{cores} threads; tokens/s = token-heads/s / {cfg.num_heads}")
    return rate, dt, cores, desc


def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = W.prefill_config()
    times, rates = [], []
    heads, tokens = 16, 2048
    for i in range(args.warmup + args.steps):
        rate, dt, cores, desc = oracle_sample(cfg, heads, tokens, seed=i)
        if i >= args.warmup:
            times.append(dt)
            rates.append(rate)
    value = float(np.mean(rates))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "global_batch": 1, "seq_len": 8192, "heads": 96, "dk": 128,
                       "dv": 128, "qkv_dtype": "bf16", "l2": "inputs larger than L2"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- CUDA arm
def _time_prefill(kda, d, out, fin, ws, stream, steps, warmup):
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    for _ in range(warmup):
        kda.prefill(*args, out=out, final_state=fin, workspace=ws, stream=stream)
    stream.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    return args, evs


def run_cuda(args, world, rank, local):
    import linear_attention_serving_chunkwise_gb300 as kda
    from linear_attention_serving_chunkwise_gb300.build import build

    if rank == 0:
        build()
    _barrier(world)
    kda.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = _peaks()
    stream = torch.cuda.Stream(device=dev)

    # ---------------- prefill: the headline step
    cfg = W.prefill_config()
    d = W.make_prefill_inputs(cfg, seed=rank, device=dev)   # one independent problem per rank
    out = torch.empty((cfg.total_tokens, cfg.num_heads, cfg.dv), dtype=torch.float32, device=dev)
    fin = torch.empty((1, cfg.num_heads, cfg.dk, cfg.dv), dtype=torch.float32, device=dev)
    desc = kda.make_desc(1, cfg.total_tokens, cfg.num_heads, cfg.dk, cfg.dv, kda.KDA_BF16)
    plan = kda.prefill_query(desc)
    ws = torch.empty(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device=dev)   # allocated once
    pargs, evs = _time_prefill(kda, d, out, fin, ws, stream, args.steps, args.warmup)
    if kda.last_device_status(stream) != kda.KDA_OK:
        raise RuntimeError("prefill reported a device error during warm-up")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()   # runs until the last leg; only samples inside the legs' windows count
    time.sleep(0.1)
    w0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        evs[i][0].record(stream)
        kda.prefill(*pargs, out=out, final_state=fin, workspace=ws, stream=stream)
        evs[i][1].record(stream)
    end.record(stream)
    stream.synchronize()
    sampler.window("prefill", w0, time.time())
    torch.cuda.synchronize()
    _barrier(world)
    if kda.last_device_status(stream) != kda.KDA_OK:
        raise RuntimeError("prefill reported a device error in the timed region")
    total_ms = _max_over_ranks(start.elapsed_time(end), world)
    launch_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    ms_per_step = total_ms / args.steps
    tokens_per_step = cfg.total_tokens * world
    value = tokens_per_step / (ms_per_step / 1e3)

    alg_bytes, alg_flops = prefill_algorithmic(cfg)
    achieved_gbs = alg_bytes / (launch_ms / 1e3) / 1e9
    achieved_tflops = alg_flops / (launch_ms / 1e3) / 1e12
    src_hash = _src_hash(PREFILL_KERNEL_SRC)
    traffic = _profiled_traffic("kda_prefill", src_hash)
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                "frac_of_nominal": achieved_gbs / NOMINAL_HBM_GBS, "nominal_gbs": NOMINAL_HBM_GBS,
                "peak_source": f"{peaks['source']} hbm_gbs (copy bandwidth)",
                "algorithmic_bytes_per_launch": alg_bytes, "kernel_launches_per_call": plan["kernel_launches"],
                "launch_ms": launch_ms,
                "kernels": PREFILL_KERNELS.get(plan["kernel_launches"], "?"),
                "timed": "CUDA events on the launching stream around each kda_prefill call (all its launches); "
                         "per-kernel shares in profiles/bench_launch_list_prefill_decode.md",
                "workspace_bytes": plan["workspace_bytes"]}
    tensor = {"achieved": achieved_tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
              "frac": achieved_tflops / peaks["bf16_tflops"], "algorithmic_flops_per_launch": alg_flops,
              "uses_tensor_cores": bool(plan["tensor_cores"]),
              "pipe_active_pct_ncu": _profiled_tensor_pipe(src_hash),
              "pipe_target_pct": 50.0,
              "pipe_note": "sm__pipe_tensor_cycles_active of the intra-chunk MMA kernels (ncu, small case, "
                           "profiles/kda_prefill_tensor_pipe.txt); null when the capture is not of this source"}

    # ---------------- end to end: kda_prefill_host from pinned host inputs to pinned host
    # outputs (out + final state), every step; the library pipelines the copies over
    # 1024-token rounds against the kernels
    host = {k: (None if v is None else v.to("cpu").pin_memory()) for k, v in d.items()}
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    host_fin = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = host_out.numel() * 4 + host_fin.numel() * 4
    e2e_steps = max(1, min(args.steps, 20))
    seg = E2E_SEGMENT_TOKENS
    hdesc = kda.make_desc(cfg.num_seqs, cfg.total_tokens, cfg.num_heads, cfg.dk, cfg.dv,
                          kda.KDA_BF16 if cfg.qkv_dtype == torch.bfloat16 else kda.KDA_F32)
    ws = torch.empty(kda.prefill_host_workspace_bytes(hdesc, seg), dtype=torch.uint8, device=dev)

    def e2e_step():
        kda.prefill_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["cu_seqlens"],
                         host["init_state"], out=host_out, final_state=host_fin, segment_tokens=seg,
                         num_seqs=cfg.num_seqs, workspace=ws, stream=stream)

    for _ in range(2):
        e2e_step()
    stream.synchronize()
    _barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    stream.synchronize()
    sampler.window("e2e", w0, time.time())
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    e2e = {"value": tokens_per_step / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
           "api": "kda_prefill_host", "segment_tokens": seg,
           "link": _link_floor(h2d, d2h, dev)}
    del host, host_out, host_fin, ws

    # ---------------- decode: 64 consecutive in-place steps
    dcfg = W.decode_config()
    dd = W.make_decode_inputs(dcfg, seed=rank, device=dev)
    state = dd["state0"]
    dout = torch.empty((dcfg.batch, dcfg.num_heads, dcfg.dv), dtype=torch.float32, device=dev)
    for s in range(3):
        kda.decode(dd["q"][s], dd["k"][s], dd["v"][s], dd["g"][s], dd["beta"][s], state, out=dout, stream=stream)
    stream.synchronize()
    devs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(dcfg.steps)]
    _barrier(world)
    w0 = time.time()
    for s in range(dcfg.steps):
        devs[s][0].record(stream)
        kda.decode(dd["q"][s], dd["k"][s], dd["v"][s], dd["g"][s], dd["beta"][s], state, out=dout, stream=stream)
        devs[s][1].record(stream)
    stream.synchronize()
    sampler.window("decode", w0, time.time())
    dstep_ms = float(np.mean([a.elapsed_time(b) for a, b in devs]))
    dstep_ms = _max_over_ranks(dstep_ms, world)
    state_bytes, all_bytes = decode_algorithmic(dcfg)
    decode = {"workload": dcfg.name, "steps": dcfg.steps, "ms_per_step": dstep_ms,
              "tokens_per_s": dcfg.batch * world / (dstep_ms / 1e3),
              "state_gbs": state_bytes / (dstep_ms / 1e3) / 1e9,
              "all_bytes_gbs": all_bytes / (dstep_ms / 1e3) / 1e9,
              "roofline": {"bound": "hbm", "achieved": all_bytes / (dstep_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": all_bytes / (dstep_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                           "frac_of_nominal": all_bytes / (dstep_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                           "traffic": _profiled_traffic("kda_decode", _src_hash(
                               ("linear_attention_serving_chunkwise_gb300/csrc/kda_decode.cu",))),
                           "algorithmic_bytes_per_launch": all_bytes},
              "gpu_launches": dcfg.steps}
    del dd, state

    # ---------------- multi-token decode: K = 4 draft tokens per sequence, same B and H
    K = 4
    mm = W.make_decode_inputs(dcfg, seed=rank, device=dev, steps=K)
    mx = {n: mm[n].transpose(0, 1).contiguous() for n in ("q", "k", "v", "g", "beta")}
    mstate = mm["state0"]
    mout = torch.empty((dcfg.batch, K, dcfg.num_heads, dcfg.dv), dtype=torch.float32, device=dev)
    mcalls = 16
    for _ in range(3):
        kda.decode_multi(mx["q"], mx["k"], mx["v"], mx["g"], mx["beta"], mstate, out=mout, stream=stream)
    stream.synchronize()
    _barrier(world)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    m0.record(stream)
    for _ in range(mcalls):
        kda.decode_multi(mx["q"], mx["k"], mx["v"], mx["g"], mx["beta"], mstate, out=mout, stream=stream)
    m1.record(stream)
    stream.synchronize()
    sampler.window("decode_multi", w0, time.time())
    mcall_ms = _max_over_ranks(m0.elapsed_time(m1) / mcalls, world)
    e_in = 2 if dcfg.qkv_dtype == torch.bfloat16 else 4
    per_head_token = e_in * (2 * dcfg.dk + dcfg.dv) + 4 * dcfg.dk + 4 + 4 * dcfg.dv
    m_bytes = dcfg.batch * dcfg.num_heads * (2 * dcfg.dk * dcfg.dv * 4 + K * per_head_token)
    decode_multi = {"workload": f"decode_multi_bf16_b{dcfg.batch}_h{dcfg.num_heads}_k{K}_d{dcfg.dk}",
                    "tokens_per_call": K, "calls": mcalls, "ms_per_call": mcall_ms,
                    "tokens_per_s": dcfg.batch * K * world / (mcall_ms / 1e3),
                    "vs_k_single_steps": (K * dstep_ms) / mcall_ms,
                    "roofline": {"bound": "hbm", "achieved": m_bytes / (mcall_ms / 1e3) / 1e9,
                                 "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": m_bytes / (mcall_ms / 1e3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                                 "frac_of_nominal": m_bytes / (mcall_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                                 "algorithmic_bytes_per_launch": m_bytes},
                    "gpu_launches": mcalls}
    del mm, mx, mstate, mout

    # ---------------- the input prologue: the same prefill from the recipe's raw draws, with q/k
    # normalisation and the g and beta parametrisations inside the kernels' loads (its own
    # workspace: the headline one was released above).  A failure here is reported in the line.
    prologue = {"workload": cfg.name + "_raw_inputs", "bits": "q/k L2 norm, g = -5 sigmoid(z), beta = sigmoid(y)"}
    try:
        draw = W.make_prefill_inputs(cfg, seed=rank, device=dev, raw=True)
        pws = torch.empty(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device=dev)
        rargs = (draw["q"], draw["k"], draw["v"], draw["g"], draw["beta"], draw["cu_seqlens"], draw["init_state"])

        def pro_call():
            kda.prefill(*rargs, out=out, final_state=fin, workspace=pws, stream=stream,
                        prologue=kda.KDA_PROLOGUE_ALL)

        for _ in range(args.warmup):
            pro_call()
        stream.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        w0 = time.time()
        p0.record(stream)
        for _ in range(args.steps):
            pro_call()
        p1.record(stream)
        stream.synchronize()
        sampler.window("prologue", w0, time.time())
        if kda.last_device_status(stream) != kda.KDA_OK:
            raise RuntimeError("prefill with the prologue reported a device error")
        pro_ms = _max_over_ranks(p0.elapsed_time(p1) / args.steps, world)
        prologue.update({"ms_per_call": pro_ms, "tokens_per_s": tokens_per_step / (pro_ms / 1e3),
                         "vs_plain_call": ms_per_step / pro_ms,
                         "roofline": {"bound": "hbm", "achieved": alg_bytes / (pro_ms / 1e3) / 1e9,
                                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": alg_bytes / (pro_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                      "frac_of_nominal": alg_bytes / (pro_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                                      "traffic": None, "algorithmic_bytes_per_launch": alg_bytes},
                         "gpu_launches": args.steps * plan["kernel_launches"]})
        del draw, rargs, pws
    except Exception as exc:   # noqa: BLE001 -- recorded in the line instead of ending the run
        prologue["error"] = f"{type(exc).__name__}: {exc}"

    # ---------------- the output gate: the headline call with gate logits z [T, H, dv] fp32
    # (out = o * sigmoid(z)), through kda_prefill_gated; 512 more bytes read per token-head
    gate = {"workload": cfg.name + "_gated", "api": "kda_prefill_gated"}
    try:
        z = W.make_gate_logits((cfg.total_tokens, cfg.num_heads, cfg.dv), seed=rank, device=dev)
        gws = torch.empty(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device=dev)

        def gate_call():
            kda.prefill(*pargs, out=out, final_state=fin, workspace=gws, stream=stream, gate=z)

        for _ in range(args.warmup):
            gate_call()
        stream.synchronize()
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        w0 = time.time()
        q0.record(stream)
        for _ in range(args.steps):
            gate_call()
        q1.record(stream)
        stream.synchronize()
        sampler.window("gate", w0, time.time())
        if kda.last_device_status(stream) != kda.KDA_OK:
            raise RuntimeError("the gated prefill reported a device error")
        gate_ms = _max_over_ranks(q0.elapsed_time(q1) / args.steps, world)
        gate_bytes = alg_bytes + cfg.total_tokens * cfg.num_heads * cfg.dv * 4
        gate.update({"ms_per_call": gate_ms, "tokens_per_s": tokens_per_step / (gate_ms / 1e3),
                     "vs_plain_call": ms_per_step / gate_ms,
                     "roofline": {"bound": "hbm", "achieved": gate_bytes / (gate_ms / 1e3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": gate_bytes / (gate_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                  "frac_of_nominal": gate_bytes / (gate_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                                  "traffic": None, "algorithmic_bytes_per_launch": gate_bytes},
                     "gpu_launches": args.steps * plan["kernel_launches"]})
        del z, gws
    except Exception as exc:   # noqa: BLE001 -- recorded in the line instead of ending the run
        gate["error"] = f"{type(exc).__name__}: {exc}"

    # ---------------- state checkpoints: the headline call with a snapshot of every (sequence,
    # head)'s state after each 512 tokens (16 slots, 100.7 MB more written per call)
    ckpt = {"workload": cfg.name + "_checkpoints", "api": "kda_prefill_checkpointed", "interval": 512, "slots": 16}
    try:
        cws = torch.empty(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device=dev)
        slots = torch.empty((1, cfg.num_heads, 16, cfg.dk, cfg.dv), dtype=torch.float32, device=dev)

        def ckpt_call():
            kda.prefill(*pargs, out=out, final_state=fin, workspace=cws, stream=stream, checkpoint_interval=512,
                        checkpoint_slots=16, checkpoints=slots)

        for _ in range(args.warmup):
            ckpt_call()
        stream.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        w0 = time.time()
        c0.record(stream)
        for _ in range(args.steps):
            ckpt_call()
        c1.record(stream)
        stream.synchronize()
        sampler.window("checkpoints", w0, time.time())
        if kda.last_device_status(stream) != kda.KDA_OK:
            raise RuntimeError("the checkpointed prefill reported a device error")
        ck_ms = _max_over_ranks(c0.elapsed_time(c1) / args.steps, world)
        ck_bytes = alg_bytes + slots.numel() * 4
        ckpt.update({"ms_per_call": ck_ms, "tokens_per_s": tokens_per_step / (ck_ms / 1e3),
                     "vs_plain_call": ms_per_step / ck_ms,
                     "roofline": {"bound": "hbm", "achieved": ck_bytes / (ck_ms / 1e3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": ck_bytes / (ck_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                                  "frac_of_nominal": ck_bytes / (ck_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                                  "traffic": None, "algorithmic_bytes_per_launch": ck_bytes},
                     "gpu_launches": args.steps * plan["kernel_launches"]})
        del cws, slots
    except Exception as exc:   # noqa: BLE001 -- recorded in the line instead of ending the run
        ckpt["error"] = f"{type(exc).__name__}: {exc}"

    # ---------------- fp32 inputs: the headline workload with q, k, v in fp32, on the CUDA-core
    # chunkwise kernel (the path of the 1e-4 bar); at most 10 timed calls, as each takes ~15 ms.
    # Its bound is the fp32 FMA pipe: 152 SMs x 128 FMA lanes x 2 flop x 2.07 GHz (maximum SM clock).
    fp32 = {"workload": cfg.name.replace("bf16", "fp32"), "kernel": "kda_prefill_simt_kernel"}
    try:
        fcfg = W.PrefillConfig(fp32["workload"], cfg.seqlens, cfg.num_heads, cfg.dk, cfg.dv, torch.float32,
                               cfg.init_state)
        fd = W.make_prefill_inputs(fcfg, seed=rank, device=dev)
        fplan = kda.prefill_query(kda.make_desc(fcfg.num_seqs, fcfg.total_tokens, fcfg.num_heads, fcfg.dk,
                                                fcfg.dv, kda.KDA_F32))
        fws = torch.empty(max(fplan["workspace_bytes"], 16), dtype=torch.uint8, device=dev)
        fargs = (fd["q"], fd["k"], fd["v"], fd["g"], fd["beta"], fd["cu_seqlens"], fd["init_state"])
        fsteps = min(args.steps, 10)

        def f32_call():
            kda.prefill(*fargs, out=out, final_state=fin, workspace=fws, stream=stream)

        for _ in range(min(args.warmup, 3)):
            f32_call()
        stream.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(world)
        w0 = time.time()
        f0.record(stream)
        for _ in range(fsteps):
            f32_call()
        f1.record(stream)
        stream.synchronize()
        sampler.window("fp32", w0, time.time())
        if kda.last_device_status(stream) != kda.KDA_OK:
            raise RuntimeError("the fp32 prefill reported a device error")
        f_ms = _max_over_ranks(f0.elapsed_time(f1) / fsteps, world)
        f_bytes, f_flops = prefill_algorithmic(fcfg)
        fp32_peak_tflops = 152 * 128 * 2 * 2.07e9 / 1e12
        fp32.update({"ms_per_call": f_ms, "tokens_per_s": tokens_per_step / (f_ms / 1e3), "calls": fsteps,
                     "vs_bf16_call": ms_per_step / f_ms,
                     "roofline": {"bound": "alu", "achieved": f_flops / (f_ms / 1e3) / 1e12,
                                  "peak": fp32_peak_tflops, "unit": "TFLOP/s",
                                  "frac": f_flops / (f_ms / 1e3) / 1e12 / fp32_peak_tflops, "traffic": None,
                                  "algorithmic_flops_per_launch": f_flops,
                                  "hbm_gbs": f_bytes / (f_ms / 1e3) / 1e9},
                     "gpu_launches": fsteps * fplan["kernel_launches"]})
        del fd, fargs, fws
    except Exception as exc:   # noqa: BLE001 -- recorded in the line instead of ending the run
        fp32["error"] = f"{type(exc).__name__}: {exc}"

    # ---------------- context parallelism emulated on this GPU: the headline sequence as two
    # token ranges (local transition and zero-start passes of both as one varlen call each, the
    # fold, the rerun from the folded states).  Three prefill passes, so slower than one call on
    # one GPU by design: it measures the scheme's cost, not a speedup.
    cp = {"workload": cfg.name + "_two_ranges", "api": "kcp.virtual_ranks_prefill", "ranks": 2}
    try:
        from linear_attention_serving_chunkwise_gb300 import kcp

        def cp_call():
            return kcp.virtual_ranks_prefill(*pargs[:5], pargs[6], ranks=2, stream=stream)

        for _ in range(3):
            cp_call()
        stream.synchronize()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cp_steps = max(3, min(args.steps, 20))
        _barrier(world)
        w0 = time.time()
        k0.record(stream)
        for _ in range(cp_steps):
            cp_call()
        k1.record(stream)
        stream.synchronize()
        sampler.window("context_parallel", w0, time.time())
        if kda.last_device_status(stream) != kda.KDA_OK:
            raise RuntimeError("the context-parallel prefill reported a device error")
        cp_ms = _max_over_ranks(k0.elapsed_time(k1) / cp_steps, world)
        cp.update({"ms_per_call": cp_ms, "tokens_per_s": tokens_per_step / (cp_ms / 1e3),
                   "vs_plain_call": ms_per_step / cp_ms, "steps": cp_steps,
                   "gpu_launches_per_call": "3 prefill calls (3 launches each at these 192 units: offsets, prep, scan), 1 kda_state_combine"})
    except Exception as exc:   # noqa: BLE001 -- recorded in the line instead of ending the run
        cp["error"] = f"{type(exc).__name__}: {exc}"
    clocks = sampler.stop()

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if plan["tensor_cores"] else "f32", "data": "synthetic",
            "config": {"workload": cfg.name, "global_batch": world, "seq_len": cfg.total_tokens,
                       "heads": cfg.num_heads, "dk": cfg.dk, "dv": cfg.dv, "qkv_dtype": "bf16",
                       "init_state": "N(0,0.02)", "l2": "inputs larger than L2 (1.41 GB per step), no flush",
                       "parallelism": f"independent problem per GPU x{world}"},
            "roofline": roofline, "tensor": tensor, "e2e": e2e, "clocks": clocks,
            "gpu_launches": args.steps * plan["kernel_launches"], "decode": decode, "decode_multi": decode_multi,
            "prologue": prologue, "gate": gate, "checkpoints": ckpt, "fp32": fp32, "context_parallel": cp}
    if rank == 0 and world == 1:
        rate, dt, cores, sdesc = oracle_sample(cfg, heads=96, tokens=8192)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sdesc,
                                "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ncu_case(case: str):
    """A small, self-contained launch for ncu captures (no timing, no JSON): the same kernels
    as the bench on inputs still larger than L2 but only a few hundred MB on the device.
      prefill: B=1, H=32, T=8192, dk=dv=128, bf16 (470 MB of inputs/outputs; the
               chunk-parallel path: chunk offsets, then the cooperative prep-and-scan kernel)
      prefill_sep: 2 sequences of 4096 tokens, H=64 (128 units: the chunk-parallel path as
               separate chunk-prep and state-scan launches, so each can be captured alone)
      prefill_one_cta: 4 sequences of 2048 tokens, H=38 (152 units, one full wave: one CTA
               per (sequence, head))
      decode:  B=64, H=96, dk=dv=128, bf16, one step (403 MB of state)
      decode_multi: the same B, H with K = 4 tokens per sequence in one call"""
    import linear_attention_serving_chunkwise_gb300 as kda
    from linear_attention_serving_chunkwise_gb300.build import build
    build()
    kda.load()
    if case == "prefill":
        cfg = W.PrefillConfig("ncu_prefill_h32_t8192", (8192,), 32, 128, 128, torch.bfloat16, "normal")
        d = W.make_prefill_inputs(cfg, seed=0, device="cuda")
        for _ in range(2):
            kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    elif case == "prefill_sep":
        cfg = W.PrefillConfig("ncu_prefill_sep_2x4096_h64", (4096,) * 2, 64, 128, 128, torch.bfloat16, "normal")
        d = W.make_prefill_inputs(cfg, seed=0, device="cuda")
        plan = kda.prefill_query(kda.make_desc(2, 8192, 64, 128, 128, kda.KDA_BF16))
        if plan["kernel_launches"] != 3:
            raise SystemExit(f"prefill_sep expected the separate launches, got {plan}")
        for _ in range(2):
            kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    elif case == "prefill_one_cta":
        cfg = W.PrefillConfig("ncu_prefill_one_cta_4x2048_h38", (2048,) * 4, 38, 128, 128, torch.bfloat16, "normal")
        d = W.make_prefill_inputs(cfg, seed=0, device="cuda")
        for _ in range(2):
            kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    elif case == "decode":
        cfg = W.DecodeConfig("ncu_decode_b64_h96", 64, 96, 128, 128, torch.bfloat16, 2)
        d = W.make_decode_inputs(cfg, seed=0, device="cuda")
        st = d["state0"]
        for s in range(2):
            kda.decode(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], st)
    else:
        cfg = W.DecodeConfig("ncu_decode_multi_b64_h96_k4", 64, 96, 128, 128, torch.bfloat16, 4)
        d = W.make_decode_inputs(cfg, seed=0, device="cuda")
        x = {n: d[n].transpose(0, 1).contiguous() for n in ("q", "k", "v", "g", "beta")}
        st = d["state0"]
        for _ in range(2):
            kda.decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], st)
    torch.cuda.synchronize()
    if kda.last_device_status() != kda.KDA_OK:
        raise SystemExit("device error")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--ncu-case", default=None,
                    choices=["prefill", "prefill_sep", "prefill_one_cta", "decode", "decode_multi"],
                    help="run one small launch pair for an ncu capture and exit")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    world, rank, local = _dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_cuda(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

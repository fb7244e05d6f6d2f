#!/usr/bin/env python3
"""Throughput of the Sparse Delta Memory write/read op on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload layer] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic input, as a
layer call runs it: the per-stream copy of the learned bank, product-key scoring and
exact top-k of both queries, the chunk plan and the fused gather / gated delta-rule
update / read (sdm_write_read with bank_init).  The default workload is the README
layer call (B=2, T=4096, 2 heads of 1024, 65536 slots from two factors of 256, W=R=64,
chunk 64, bf16 activations, fp32 bank).  Prints one JSON line (rank 0).

Multi-GPU (torchrun): every rank runs its own streams (weak scaling, no collective on
the data path); the timed region is bracketed by barriers and the slowest rank's time
is reported.  --impl reference times the CPU oracle on the host instead (rank 0 only).
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import sdm_inputs  # noqa: E402

METRIC = "SDM write/read tokens/s per layer on 1 GB300; achieved HBM GB/s vs roofline"
UNIT = "tokens/s"
WORKLOADS = {"layer": "layer", "train_fwd": "train_fwd", "three_factor": "three_factor",
             "decode": "decode", "tiny": "tiny", "train": "train_fwd", "readme_layer": "layer",
             "layer_train": "train_fwd"}
README_DIM = 2048          # the README usage example's model width (dim = num_heads * d_v)
KERNEL_SOURCES = ("sdm_write_read.cu", "sdm_write_read_f32_f32.cu", "sdm_write_read_f32_bf16.cu",
                  "sdm_write_read_bf16_f32.cu", "sdm_write_read_bf16_bf16.cu", "sdm_wr_kernel.cuh",
                  "sdm_delta.cuh", "sdm_common.cuh", "sdm_internal.h")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(cfg, rank: int) -> int:
    """Seed of a rank's inputs: every rank runs its own streams (independent problems)."""
    return cfg.seed + 7919 * rank


def rank_streams(B: int, H: int, rank: int, world: int) -> list:
    """The global streams (b, h) rank ``rank`` runs: the job's batch is world*B elements and
    rank r holds elements r*B .. r*B + B - 1, every head of each (its inputs are drawn with
    rank_seed, so they are that slice of the global batch)."""
    return [(rank * B + b, h) for b in range(B) for h in range(H)]


def max_over_ranks(x: float, pg, device) -> float:
    """The largest of the ranks' values (a time): the whole job is as slow as its slowest rank."""
    if pg is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units per second of all ranks together, timed by the slowest rank's ``ms``."""
    return units_per_rank * world / (ms / 1e3)


def workload_desc(cfg) -> str:
    dims = "x".join(str(n) for n in cfg.factor_dims)
    return (f"{cfg.name}: B={cfg.B} T={cfg.T} H={cfg.H} d_v={cfg.d_v} factors={dims} "
            f"(N={cfg.N}/head) d_sub={cfg.d_sub} W={cfg.W} R={cfg.R} chunk={cfg.chunk_size} "
            f"acts={cfg.act_dtype} bank={cfg.bank_dtype}")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gated_delta_rule_factor_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per write/read launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"write_read_{workload}_traffic.txt")
    rec = {}
    try:
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
    except OSError:
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return int(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


_ORACLE_TIMER = r"""
import json, sys, time
sys.path.insert(0, %(root)r)
import numpy as np
import sdm_inputs, oracle
cfg = sdm_inputs.CONFIGS[%(workload)r]
budget = %(budget)f
T_max = min(cfg.T, %(t_max)d)
d = sdm_inputs.make_inputs(cfg, T=T_max)
f64 = lambda t: t.float().double().numpy()
q_w, q_r, k_val, gates, subkeys = (f64(d[k]) for k in ("q_w", "q_r", "k_val", "gates", "subkeys"))
banks = [f64(d["bank_init"][h]).copy() for h in range(cfg.H)]    # batch element 0, every head
kw = dict(factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, W=cfg.W, R=cfg.R,
          act_dtype=cfg.act_dtype, bank_dtype=cfg.bank_dtype)
done, spent, per, chunks = 0, 0.0, %(per)d, []
while done + per <= T_max and (spent < budget or done == 0):
    t0 = time.perf_counter()
    for h in range(cfg.H):
        sl = slice(done, done + per)
        oracle.run_stream(banks[h], q_w[0, sl, h], q_r[0, sl, h], k_val[0, sl, h], gates[0, sl, h],
                          subkeys[h], **kw)
    chunks.append(time.perf_counter() - t0)
    spent += chunks[-1]
    done += per
print(json.dumps({"tokens": done, "seconds": spent, "heads": cfg.H, "chunk_seconds": chunks}))
"""


def _time_oracle(workload: str, budget_s: float, t_max: int, per: int) -> dict:
    code = _ORACLE_TIMER % {"root": ROOT, "workload": workload, "budget": budget_s, "t_max": t_max,
                            "per": per}
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def chunk_collision_rate(idx_w, idx_r, chunk: int) -> float:
    """1 - (distinct rows / references), summed over every chunk of every stream."""
    import numpy as np
    B, T, H, _ = idx_w.shape
    refs = distinct = 0
    for b in range(B):
        for h in range(H):
            for t0 in range(0, T, chunk):
                ids = np.concatenate([idx_w[b, t0:t0 + chunk, h].ravel(), idx_r[b, t0:t0 + chunk, h].ravel()])
                refs += ids.size
                distinct += np.unique(ids).size
    return 1.0 - distinct / max(refs, 1)


def cpu_baseline(workload: str, budget_s: float = 15.0) -> dict:
    """Time the CPU oracle (one thread, fresh process) on a bounded sample of the workload."""
    try:
        res = _time_oracle(workload, budget_s, t_max=4096, per=8)
    except Exception as e:  # reported, not fatal
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {e}"[:300]}
    return {"value": res["tokens"] / res["seconds"], "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"the first {res['tokens']} tokens of batch element 0 through every head "
                       f"({res['heads']}), state carried token to token from the learned table; "
                       f"{res['seconds']:.1f} s of CPU work, single-threaded numpy (BLAS threads = 1)")}


def reference_arm(args, cfg, rank, world):
    """--impl reference: the CPU oracle on the host cores, same metric, unit and config.

    Each step runs a bounded sample (a few tokens of batch element 0 through every head,
    the state carried from step to step); the whole run stays within a few minutes."""
    if rank != 0:
        return 0
    per = 2 if cfg.N >= 65536 else 8
    n_steps = min(args.warmup + args.steps, cfg.T // per)
    res = _time_oracle(WORKLOADS[args.workload], budget_s=1e30, t_max=n_steps * per, per=per)
    timed = res["chunk_seconds"][args.warmup:]
    tokens = per * len(timed)
    dt = max(sum(timed), 1e-9)
    value = tokens / dt
    steps = tokens // per
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(cfg)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{per} tokens of batch element 0 through all {cfg.H} heads per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="layer", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override the workload's T (smaller cases for profiler captures)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's B (smaller cases for profiler captures)")
    ap.add_argument("--wr-slice", type=int, default=0, choices=[0, 32, 128, 256],
                    help="tuning: force the write/read kernel's row slice per CTA in bytes (0 = automatic)")
    ap.add_argument("--wr-stage", type=int, default=0,
                    help="tuning: cap the write/read kernel's stage length in tokens (0 = automatic)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local = dist_env()
    cfg = sdm_inputs.CONFIGS[WORKLOADS[args.workload]]
    if args.seq_len > 0 and cfg.T > 1:
        cfg = dataclasses.replace(cfg, T=args.seq_len)
    if args.batch > 0:
        cfg = dataclasses.replace(cfg, B=args.batch)

    if args.impl == "reference":
        return reference_arm(args, cfg, rank, world)

    import gated_delta_rule_factor_gb300 as sdm

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.wr_slice or args.wr_stage:
        sdm.test_force_write_read_layout(args.wr_slice, args.wr_stage)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    if cfg.T == 1:
        return bench_decode(args, cfg, sdm, dev, rank, world, barrier, pg)
    if args.workload == "train":
        return bench_train(args, cfg, sdm, dev, rank, world, barrier, pg)
    if args.workload == "readme_layer":
        return bench_readme_layer(args, cfg, sdm, dev, rank, world, barrier, pg)
    if args.workload == "layer_train":
        return bench_layer_train(args, cfg, sdm, dev, rank, world, barrier, pg)

    d = sdm_inputs.make_inputs(cfg, seed=rank_seed(cfg, rank))
    g = {k: v.to(dev) for k, v in d.items()}
    B, T, H = cfg.B, cfg.T, cfg.H
    bank = torch.empty((B, H, cfg.N, cfg.d_v), dtype=g["bank_init"].dtype, device=dev)
    y = torch.empty_like(g["k_val"])
    shape = sdm.make_shape(B=B, T=T, H=H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                           W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size,
                           act_dtype=0 if cfg.act_dtype == "f32" else 1,
                           bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    ws = torch.empty(sdm.write_read_workspace_size(shape), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, cfg.chunk_size,
                           cfg.W, cfg.R, factor_dims=cfg.factor_dims, bank_init=g["bank_init"], y=y,
                           workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    barrier()
    assert sdm.last_device_error(ws) == 0

    # ---- device-resident timed region
    launches0 = sdm.launch_count()
    sdm.profile_begin()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
    kt = sdm.profile_end()
    launches = sdm.launch_count() - launches0
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
    value = whole_job_rate(B * T * args.steps, world, ms)

    # ---- roofline of the dominant kernel (fused gather / update / read)
    sb = 4 if cfg.bank_dtype == "f32" else 2
    wr_launches, wr_ms = kt["write_read"]
    wr_avg_s = wr_ms / max(wr_launches, 1) / 1e3
    alg_bytes = B * T * H * (cfg.W + cfg.R) * cfg.d_v * sb
    peak, peak_kind = peaks()
    achieved = alg_bytes / wr_avg_s / 1e9
    traffic = recorded_traffic(args.workload)
    copy_bytes = 2 * B * H * cfg.N * cfg.d_v * sb
    step_alg = alg_bytes + copy_bytes

    # ---- within-chunk collision rate: 1 - distinct rows / references per chunk of a stream
    idx_w = torch.empty((B, T, H, cfg.W), dtype=torch.int32, device=dev)
    idx_r = torch.empty((B, T, H, cfg.R), dtype=torch.int32, device=dev)
    sdm.sdm_write_read(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, cfg.chunk_size,
                       cfg.W, cfg.R, factor_dims=cfg.factor_dims, bank_init=g["bank_init"], y=y, idx_w=idx_w,
                       idx_r=idx_r, workspace=ws, stream=stream)
    collision = chunk_collision_rate(idx_w.cpu().numpy(), idx_r.cpu().numpy(), cfg.chunk_size)

    # ---- end to end through the public API with host buffers: every step copies its
    # inputs from pinned host memory and its y back, pipelined the way a serving loop
    # would run it: two device buffer sets, step i+1's inputs upload on one copy stream
    # while step i computes, and step i's y downloads on another during step i+1
    e2e = None
    if not args.no_e2e:
        host = {k: d[k].pin_memory() for k in ("q_w", "q_r", "k_val", "gates")}
        y_hosts = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = y_hosts[0].numel() * y_hosts[0].element_size()
        bufs = [{k: torch.empty_like(g[k]) for k in host} for _ in range(2)]
        ys = [torch.empty_like(y) for _ in range(2)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        ev_back = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            k = i % 2
            if used[k]:
                up.wait_event(ev_out[k])          # step i-2 is done with these inputs
            with torch.cuda.stream(up):
                for name, v in host.items():
                    bufs[k][name].copy_(v, non_blocking=True)
            ev_in[k].record(up)
            stream.wait_event(ev_in[k])
            if used[k]:
                stream.wait_event(ev_back[k])     # step i-2's y has left ys[k]
            sdm.sdm_write_read(bufs[k]["q_w"], bufs[k]["q_r"], bufs[k]["k_val"], bufs[k]["gates"], g["subkeys"],
                               bank, cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                               bank_init=g["bank_init"], y=ys[k], workspace=ws, stream=stream)
            ev_out[k].record(stream)
            down.wait_event(ev_out[k])
            with torch.cuda.stream(down):
                y_hosts[k].copy_(ys[k], non_blocking=True)
            ev_back[k].record(down)
            used[k] = True

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e_steps = max(10, args.steps // 3)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)
        for i in range(e_steps):
            e2e_step(i)
        for k in range(2):
            stream.wait_event(ev_back[k])
        e1.record(stream)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1), pg, dev)
        e2e = {"value": whole_job_rate(B * T * e_steps, world, ems), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "pipelining": "two device buffer sets; inputs of step i+1 upload and y of step i-1 downloads "
                             "on copy streams while step i computes"}

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "parallelism": f"streams sharded, {world} independent ranks",
                   "global_batch": B * world,
                   "l2": "inputs larger than L2: the 1 GiB bank is rewritten from the learned table every step",
                   "step": "bank copy + scoring/top-k + chunk plan + fused write/read",
                   "chunk_collision_rate": collision},
        "roofline_2w_r": {"note": "written rows counted as read and written: B*T*H*(2W+R)*d_v*elem",
                          "achieved": alg_bytes * (2 * cfg.W + cfg.R) / (cfg.W + cfg.R) / wr_avg_s / 1e9,
                          "frac": alg_bytes * (2 * cfg.W + cfg.R) / (cfg.W + cfg.R) / wr_avg_s / 1e9 / peak},
        "roofline": {"bound": "hbm", "kernel": "write_read", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "launch_ms": wr_avg_s * 1e3},
        "step_roofline": {"algorithmic_bytes": step_alg, "achieved_gbs": step_alg / (ms / args.steps / 1e3) / 1e9,
                          "frac": step_alg / (ms / args.steps / 1e3) / 1e9 / peak},
        "kernels_ms_per_step": {k: v[1] / max(v[0], 1) * (v[0] / args.steps) for k, v in kt.items() if v[0]},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def bench_train(args, cfg, sdm, dev, rank, world, barrier, pg):
    """Training step of the 32K-token shape: the forward with a snapshot of the rows each
    token overwrites (sdm_write_read_train, bank reset from the learned table), then the
    deterministic sparse backward (sdm_write_read_backward) with dL/dy drawn once and
    dL/d(final bank) = 0 (a torch fill of the gradient table each step)."""
    d = sdm_inputs.make_inputs(cfg, seed=rank_seed(cfg, rank))
    gr = sdm_inputs.make_grad_inputs(cfg, seed=rank_seed(cfg, rank), dbank=False)
    g = {k: v.to(dev) for k, v in d.items()}
    dy = gr["dy"].to(dev)
    B, T, H = cfg.B, cfg.T, cfg.H
    bank = torch.empty((B, H, cfg.N, cfg.d_v), dtype=g["bank_init"].dtype, device=dev)
    dbank = torch.zeros((B, H, cfg.N, cfg.d_v), dtype=torch.float32, device=dev)
    shape = sdm.make_shape(B=B, T=T, H=H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                           W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size,
                           act_dtype=0 if cfg.act_dtype == "f32" else 1,
                           bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    ws = torch.empty(sdm.write_read_workspace_size(shape), dtype=torch.uint8, device=dev)
    bws = torch.empty(sdm.backward_workspace_size(shape), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # a bfloat16 snapshot holds a bfloat16 bank exactly (half the bytes of a float32 one)
    snap_dt = torch.bfloat16 if cfg.bank_dtype == "bf16" else torch.float32
    saved = None
    grads = None

    def step():
        nonlocal saved, grads
        saved = sdm.sdm_write_read_train(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank,
                                         cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims,
                                         bank_init=g["bank_init"], snapshot_dtype=snap_dt, saved=saved,
                                         workspace=ws, stream=stream)
        dbank.zero_()
        grads = sdm.sdm_write_read_backward(g["q_w"], g["q_r"], g["k_val"], g["gates"], g["subkeys"], bank, dy,
                                            saved, cfg.W, cfg.R, factor_dims=cfg.factor_dims, dbank=dbank,
                                            grads=grads, workspace=bws, stream=stream)
        grads.pop("workspace", None)

    for _ in range(args.warmup):
        step()
    barrier()
    assert sdm.last_device_error(ws) == 0 and sdm.last_device_error(bws) == 0

    launches0 = sdm.launch_count()
    sdm.profile_begin()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
    kt = sdm.profile_end()
    launches = sdm.launch_count() - launches0
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
    value = whole_job_rate(B * T * args.steps, world, ms)

    sb = 4 if cfg.bank_dtype == "f32" else 2
    se = 2 if snap_dt == torch.bfloat16 else 4
    rows = B * T * H
    # per token and column: forward W+R rows (+ the W snapshot rows written); backward
    # reads the R read rows and the W snapshot rows, reads and writes the float32 gradient
    # rows of both lists and writes the W restored rows
    fwd_bytes = rows * cfg.d_v * ((cfg.W + cfg.R) * sb + cfg.W * se)
    sweep_bytes = rows * cfg.d_v * (cfg.R * sb + 2 * 4 * (cfg.W + cfg.R) + cfg.W * se + cfg.W * sb)
    peak, peak_kind = peaks()
    per = {}
    for name, nbytes in (("write_read", fwd_bytes), ("bwd_sweep", sweep_bytes)):
        n, t = kt[name]
        avg = t / max(n, 1) / 1e3
        per[name] = {"bound": "hbm", "kernel": name, "achieved": nbytes / avg / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": nbytes / avg / 1e9 / peak, "traffic": None, "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": nbytes, "launch_ms": avg * 1e3}
    dominant = max(per, key=lambda k: per[k]["launch_ms"])
    if rank != 0:
        return 0
    line = {
        "metric": "SDM training step (forward with snapshot + deterministic sparse backward) tokens/s per layer "
                  "on 1 GB300", "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(cfg) + ", forward + backward",
                   "snapshot_dtype": "bf16" if se == 2 else "f32",
                   "l2": "inputs larger than L2: the bank is rewritten from the learned table every step",
                   "step": "bank copy + scoring/top-k + chunk plan + write/read with snapshot + backward "
                           "(flags, reverse sweep, column sums + softmax + dq, sub-key gradient); dL/d(final bank) "
                           "zeroed by a torch fill"},
        "roofline": per[dominant],
        "rooflines": per,
        "kernels_ms_per_step": {k: v[1] / max(v[0], 1) * (v[0] / args.steps) for k, v in kt.items() if v[0]},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_readme_layer(args, cfg, sdm, dev, rank, world, barrier, pg):
    """The README call: the SDM layer forward around the op (x [B, T, dim] -> [B, T, dim],
    dim = 2048, the bank reset from the learned table every call), through
    sdm_layer_forward: the cuBLASLt projections, the gates kernel, the op, the output
    projection."""
    L = sdm_inputs.make_layer_inputs(cfg, README_DIM, seed=rank_seed(cfg, rank))
    g = {k: v.to(dev) for k, v in L.items()}
    B, T, H = cfg.B, cfg.T, cfg.H
    bank = torch.empty((B, H, cfg.N, cfg.d_v), dtype=g["bank_init"].dtype, device=dev)
    out = torch.empty_like(g["x"])
    shape = sdm.make_shape(B=B, T=T, H=H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                           W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size,
                           act_dtype=0 if cfg.act_dtype == "f32" else 1,
                           bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    ws = torch.empty(sdm.layer_workspace_size(shape, README_DIM), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        sdm.sdm_layer_forward(g["x"], g["w_qw"], g["w_qr"], g["w_v"], g["w_g"], g["w_o"], g["subkeys"], bank,
                              cfg.chunk_size, cfg.W, cfg.R, factor_dims=cfg.factor_dims, bank_init=g["bank_init"],
                              out=out, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    barrier()
    assert sdm.last_device_error(ws) == 0
    launches0 = sdm.launch_count()
    sdm.profile_begin()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
    kt = sdm.profile_end()
    launches = sdm.launch_count() - launches0
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
    value = whole_job_rate(B * T * args.steps, world, ms)
    sb = 4 if cfg.bank_dtype == "f32" else 2
    alg = B * T * H * (cfg.W + cfg.R) * cfg.d_v * sb
    n, t = kt["write_read"]
    avg = t / max(n, 1) / 1e3
    peak, peak_kind = peaks()
    gemm_flop = 2 * B * T * README_DIM * (2 * H * cfg.F * cfg.d_sub + 2 * H * cfg.d_v)
    gn, gt = kt["layer_gemm"]
    if rank != 0:
        return 0
    line = {
        "metric": "SDM layer forward (README call) tokens/s on 1 GB300", "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(cfg) + f", layer dim={README_DIM}",
                   "step": "query/value projections (cuBLASLt) + gates kernel + bank copy + scoring/top-k + plan "
                           "+ write/read + output projection (cuBLASLt)"},
        "roofline": {"bound": "hbm", "kernel": "write_read", "achieved": alg / avg / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": alg / avg / 1e9 / peak, "traffic": None, "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": alg, "launch_ms": avg * 1e3},
        "projections": {"flop_per_step": gemm_flop, "ms_per_step": gt / args.steps,
                        "tflops": gemm_flop / (gt / args.steps / 1e3) / 1e12 if gt else None},
        "kernels_ms_per_step": {k: v[1] / args.steps for k, v in kt.items() if v[0]},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_layer_train(args, cfg, sdm, dev, rank, world, barrier, pg):
    """One SDM layer forward + backward at 32K tokens per step (the pages' layer benchmark
    shape: dim 2048, 2 heads, 65536 slots per head, W = R = 64, bf16, B=8 T=4096): the
    training forward (projections, gates, the op with a bf16 snapshot, output projection)
    and the layer backward (the products, the op's backward, the gradient concatenation,
    the learned table's batch sum), dL/dout drawn once, dL/d(final bank) = 0."""
    L = sdm_inputs.make_layer_inputs(cfg, README_DIM, seed=rank_seed(cfg, rank))
    g = {k: v.to(dev) for k, v in L.items()}
    B, T, H = cfg.B, cfg.T, cfg.H
    gen = torch.Generator(device="cpu")
    gen.manual_seed(rank_seed(cfg, rank) + 77)
    dout = torch.randn(B, T, README_DIM, generator=gen).to(g["x"].dtype).to(dev)
    bank = torch.empty((B, H, cfg.N, cfg.d_v), dtype=g["bank_init"].dtype, device=dev)
    dbank = torch.zeros((B, H, cfg.N, cfg.d_v), dtype=torch.float32, device=dev)
    shape = sdm.make_shape(B=B, T=T, H=H, factor_dims=cfg.factor_dims, d_sub=cfg.d_sub, d_v=cfg.d_v,
                           W=cfg.W, R=cfg.R, chunk_size=cfg.chunk_size,
                           act_dtype=0 if cfg.act_dtype == "f32" else 1,
                           bank_dtype=0 if cfg.bank_dtype == "f32" else 1)
    ws = torch.empty(sdm.layer_workspace_size(shape, README_DIM), dtype=torch.uint8, device=dev)
    bws = torch.empty(sdm.layer_backward_workspace_size(shape, README_DIM), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    snap_dt = torch.bfloat16 if cfg.bank_dtype == "bf16" else torch.float32
    state = {"saved": None, "grads": None}
    out = torch.empty_like(g["x"])

    def step():
        _, state["saved"] = sdm.sdm_layer_forward_train(
            g["x"], g["w_qw"], g["w_qr"], g["w_v"], g["w_g"], g["w_o"], g["subkeys"], bank, cfg.chunk_size, cfg.W,
            cfg.R, factor_dims=cfg.factor_dims, bank_init=g["bank_init"], snapshot_dtype=snap_dt, out=out,
            saved=state["saved"], workspace=ws, stream=stream)
        dbank.zero_()
        grads = sdm.sdm_layer_backward(g["x"], g["w_qw"], g["w_qr"], g["w_v"], g["w_g"], g["w_o"], g["subkeys"],
                                       bank, dout, state["saved"], cfg.chunk_size, cfg.W, cfg.R,
                                       factor_dims=cfg.factor_dims, dbank=dbank, grads=state["grads"],
                                       workspace=bws, stream=stream)
        grads.pop("workspace", None)
        grads.pop("bank", None)
        state["grads"] = grads

    for _ in range(args.warmup):
        step()
    barrier()
    assert sdm.last_device_error(ws) == 0 and sdm.last_device_error(bws) == 0
    launches0 = sdm.launch_count()
    sdm.profile_begin()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
    kt = sdm.profile_end()
    launches = sdm.launch_count() - launches0
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
    value = whole_job_rate(B * T * args.steps, world, ms)
    sb = 4 if cfg.bank_dtype == "f32" else 2
    se = 2 if snap_dt == torch.bfloat16 else 4
    rows = B * T * H
    sweep_bytes = rows * cfg.d_v * (cfg.R * sb + 2 * 4 * (cfg.W + cfg.R) + cfg.W * se + cfg.W * sb)
    n, t = kt["bwd_sweep"]
    avg = t / max(n, 1) / 1e3
    peak, peak_kind = peaks()
    dq, dv = H * cfg.F * cfg.d_sub, H * cfg.d_v
    gemm_flop = 2 * B * T * README_DIM * (2 * dq + dv) * 3 + 2 * B * T * README_DIM * dv * 3
    gn, gt = kt["layer_gemm"]
    if rank != 0:
        return 0
    line = {
        "metric": "SDM layer forward + backward tokens/s at 32K tokens per step on 1 GB300", "value": value,
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(cfg) + f", layer dim={README_DIM}, forward + backward",
                   "snapshot_dtype": "bf16" if se == 2 else "f32",
                   "step": "training forward (projections, gates, op with snapshot, output projection) + layer "
                           "backward (products, op backward, gradient concatenation, batch sum); dL/d(final bank) "
                           "zeroed by a torch fill"},
        "roofline": {"bound": "hbm", "kernel": "bwd_sweep", "achieved": sweep_bytes / avg / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": sweep_bytes / avg / 1e9 / peak, "traffic": None,
                     "peak_source": peak_kind, "algorithmic_bytes_per_launch": sweep_bytes, "launch_ms": avg * 1e3},
        "products": {"flop_per_step": gemm_flop, "ms_per_step": gt / args.steps,
                     "tflops": gemm_flop / (gt / args.steps / 1e3) / 1e12 if gt else None},
        "kernels_ms_per_step": {k: v[1] / args.steps for k, v in kt.items() if v[0]},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "e2e": None,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_decode(args, cfg, sdm, dev, rank, world, barrier, pg):
    """Decode workload: B streams, one token per step, donated (in place) state."""
    steps_total = args.warmup + args.steps
    d = sdm_inputs.make_decode_inputs(cfg, steps=min(steps_total, 64), seed=rank_seed(cfg, rank))
    g = {k: v.to(dev) for k, v in d.items()}
    state = g["bank"].clone()
    donate = os.environ.get("SDM_DECODE_COPY", "0") != "1"
    stream = torch.cuda.current_stream(dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    y = torch.empty_like(g["k_val"][:, 0])
    nT = g["q_w"].shape[1]
    per_step = [tuple(g[k][:, t].contiguous() for k in ("q_w", "q_r", "k_val", "gates")) for t in range(nT)]

    def step(i):
        nonlocal state
        _, state = sdm.sdm_decode_step(*per_step[i % nT], g["subkeys"], state, cfg.W, cfg.R,
                                       factor_dims=cfg.factor_dims, donate=donate, y=y, workspace=ws,
                                       stream=stream)

    for i in range(args.warmup):
        step(i)
    barrier()
    launches0 = sdm.launch_count()
    sdm.profile_begin()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier()
        ev0.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        ev1.record(stream)
        barrier()
    kt = sdm.profile_end()
    ms = max_over_ranks(ev0.elapsed_time(ev1), pg, dev)
    value = whole_job_rate(cfg.B * args.steps, world, ms)
    launches = sdm.launch_count() - launches0
    sb = 4 if cfg.bank_dtype == "f32" else 2
    alg = cfg.B * cfg.H * (cfg.W + cfg.R) * cfg.d_v * sb + (0 if donate else 2 * cfg.B * cfg.H * cfg.N * cfg.d_v * sb)

    # the same donated steps replayed from one CUDA graph of nT steps (no per-call host
    # work or launch gaps); the copying form is left out: every captured step would keep
    # its own successor table alive in the graph's memory pool
    graph = None
    if donate:
        def gstep(i):
            nonlocal state
            _, state = sdm.sdm_decode_step(*per_step[i % nT], g["subkeys"], state, cfg.W, cfg.R,
                                           factor_dims=cfg.factor_dims, donate=True, y=y, workspace=ws)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            for i in range(nT):
                gstep(i)
        cg.replay()
        reps = max(1, args.steps // nT)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        g0.record(stream)
        for _ in range(reps):
            cg.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        gms = max_over_ranks(g0.elapsed_time(g1), pg, dev) / (reps * nT)
        graph = {"ms_per_step": gms, "value": whole_job_rate(cfg.B, world, gms), "unit": UNIT,
                 "steps": reps * nT, "steps_per_graph": nT}
    n, kms = kt["decode"]
    achieved = alg / (kms / max(n, 1) / 1e3) / 1e9
    peak, peak_kind = peaks()
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "donate": donate},
            "roofline": {"bound": "hbm", "kernel": "decode", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_kind},
            "gpu_launches": launches, "clocks": clk.summary(), "graph": graph}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())

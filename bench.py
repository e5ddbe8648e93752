"""Benchmark of the fused attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * attn_fwd on the causal prefill workload (B=4, Hq=Hkv=16, T=2048, D=128,
    bf16 N(0,1), scale 1/sqrt(128)) -- its TFLOP/s is the headline ``value``;
  * paged_attn_decode on the paged workload (64 requests x 1 token, Hq=12,
    Hkv=2, D=128, 16-token blocks, lengths U[512, 8192], random block tables)
    -- reported in ``paged_decode`` as KV GB/s.
Inputs are resident in HBM before the timed region; L2 is flushed (a 512 MiB
write) before every step, outside the kernel events.  Kernel time is taken with
CUDA events on the launching stream.  ``e2e`` repeats the prefill metric with
host (pinned) buffers: the H2D copy of q/k/v and the D2H copy of O and LSE sit
inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
device (independent replicas, weak scaling); the max time over ranks is used.
"""

from __future__ import annotations

import argparse
import hashlib
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "attn fwd TFLOP/s & % bf16 tensor peak; paged-decode KV GB/s & % HBM peak"
PREFILL = synth.CONFIGS["prefill_mha_causal"]
DECODE = synth.CONFIGS["paged_decode"]
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_name():
    return (f"causal prefill MHA B={PREFILL.B} Hq=Hkv={PREFILL.Hq} T={PREFILL.T} D={PREFILL.D} "
            f"bf16 + paged decode {DECODE.num_seqs} req x1 token Hq={DECODE.Hq} Hkv={DECODE.Hkv} "
            f"D={DECODE.D} block_size={DECODE.block_size} L~U[{DECODE.len_lo},{DECODE.len_hi}]")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_flashattention_fwd_03_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        ent = d[kernel]
        if ent.get("source_sha") != kernel_source_sha():
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# --------------------------------------------------------------------------- #
# clocks sampled during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- #
# CPU baseline: the fp64 oracle on a bounded sample
# --------------------------------------------------------------------------- #
def oracle_prefill_sample(q, k, v, target_s: float, seed: int):
    """Times the oracle on random rows of the prefill workload; returns (TFLOP/s, info)."""
    import oracle
    lib = oracle.load()
    cfg = PREFILL
    # calibration on a small sample, then a sample sized for ~target_s
    n = 64
    while True:
        rows = np.sort(synth.uniform_ints(seed, n, 0, cfg.B * cfg.Hq * cfg.T - 1))
        t0 = time.perf_counter()
        oracle.attn_rows(q, k, v, cfg.causal, cfg.softmax_scale, rows, lib=lib)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= cfg.B * cfg.Hq * cfg.T:
            break
        n = int(min(cfg.B * cfg.Hq * cfg.T, max(2 * n, n * target_s / max(dt, 1e-3) * 1.05)))
    i = rows % cfg.T
    vis = (i + 1) if cfg.causal else np.full_like(i, cfg.T)
    flops = float(np.sum(4.0 * vis * cfg.D))  # q.k and p.v multiply-adds of each sampled row
    return flops / dt / 1e12, {"rows": int(n), "seconds": dt, "flops": flops,
                               "cores": oracle.num_threads(lib)}


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor(values, dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def aggregate_value(flops_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank does the same work; time is the slowest rank's."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def run_ours(args, rank, world, local_rank):
    import torch
    import attention_flashattention_fwd_03_gb300 as gb
    gb.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    # ---- inputs (seeded, resident in HBM) ----
    qn, kn, vn = synth.prefill_inputs(PREFILL)
    q, k, v = to_dev(qn), to_dev(kn), to_dev(vn)
    o = torch.empty_like(q)
    lse = torch.empty((PREFILL.B, PREFILL.Hq, PREFILL.T), dtype=torch.float32, device=dev)
    pg = synth.paged_inputs(DECODE)
    dq, dk, dv = to_dev(pg.q), to_dev(pg.k_pool), to_dev(pg.v_pool)
    dbt, dsl = i32(pg.block_table), i32(pg.seq_lens)
    do = torch.empty_like(dq)
    dlse = torch.empty((DECODE.num_seqs, DECODE.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(gb.paged_attn_decode_workspace_size(DECODE.num_seqs, DECODE.Hq, DECODE.D,
                                                         pg.max_seq_len), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def prefill():
        gb.attn_fwd(q, k, v, causal=True, scale=PREFILL.softmax_scale, out=o, lse=lse)

    def decode():
        gb.paged_attn_decode(dq, dk, dv, dbt, dsl, pg.max_seq_len, scale=DECODE.softmax_scale,
                             out=do, lse=dlse, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        prefill()
        decode()
    torch.cuda.synchronize()
    st, flags = gb.attn_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags} after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        prefill()
        ev[i][1].record(stream)
        decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    t_pre = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    t_dec = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    launches = args.steps * 3  # 1 prefill kernel + split + merge per step
    st, flags = gb.attn_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags} after timing")

    # ---- e2e: host buffers, copies inside the timed region ----
    hq = torch.from_numpy(qn.view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = torch.from_numpy(kn.view(np.int16)).view(torch.bfloat16).pin_memory()
    hv = torch.from_numpy(vn.view(np.int16)).view(torch.bfloat16).pin_memory()
    ho = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))
    e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
    for i in range(-2, e2e_steps):
        flush.zero_()
        if i >= 0:
            e_ev[i][0].record(stream)
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        prefill()
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)
        if i >= 0:
            e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_e2e = [e_ev[i][0].elapsed_time(e_ev[i][1]) for i in range(e2e_steps)]
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2
    d2h = ho.numel() * 2 + hl.numel() * 4

    # ---- aggregate over ranks ----
    ms_pre = statistics.mean(t_pre)
    ms_dec = statistics.mean(t_dec)
    ms_e2e = statistics.mean(t_e2e)
    ms_pre, ms_dec, ms_e2e, wall = max_over_ranks([ms_pre, ms_dec, ms_e2e, wall], dev)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, info = oracle_prefill_sample(qn, kn, vn, args.cpu_seconds, PREFILL.seed + 77)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": info["cores"], "kind": "oracle",
               "sample": (f"{info['rows']} random query rows of the prefill workload "
                          f"({info['flops'] / 1e9:.1f} GFLOP of q.k and p.v in fp64) "
                          f"in {info['seconds']:.1f} s")}
    return dict(ms_pre=ms_pre, ms_dec=ms_dec, ms_e2e=ms_e2e, wall=wall, clocks=clocks,
                launches=launches, h2d=h2d, d2h=d2h, cpu=cpu,
                kv_bytes=pg.kv_bytes(DECODE.Hkv, DECODE.D),
                dec_other_bytes=(pg.q.nbytes * 2 + DECODE.num_seqs * DECODE.Hq * 4
                                 + 4 * int(sum(-(-int(L) // 16) for L in pg.seq_lens))
                                 + pg.seq_lens.nbytes),
                t_pre=t_pre, t_dec=t_dec)


def report_ours(args, res, world):
    peaks, src = load_peaks()
    flops = PREFILL.flops()
    tf_rank = flops / (res["ms_pre"] * 1e-3) / 1e12
    value = aggregate_value(flops, res["ms_pre"], world)
    frac = tf_rank / peaks["bf16_tflops"]
    dec_bytes = res["kv_bytes"] + res["dec_other_bytes"]
    gbs = dec_bytes / (res["ms_dec"] * 1e-3) / 1e9
    e2e_tf = world * flops / (res["ms_e2e"] * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(res["ms_pre"] + res["ms_dec"], 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; paged pool with random block tables)",
        "config": {
            "workload": workload_name(),
            "prefill": {"B": PREFILL.B, "Hq": PREFILL.Hq, "Hkv": PREFILL.Hkv, "T": PREFILL.T,
                        "D": PREFILL.D, "causal": True, "flops_per_step": flops,
                        "flop_convention": "4*B*Hq*T^2*D/2 (causal half)",
                        "flops_exact_causal": PREFILL.flops_exact()},
            "decode": {"num_seqs": DECODE.num_seqs, "Hq": DECODE.Hq, "Hkv": DECODE.Hkv,
                       "D": DECODE.D, "block_size": DECODE.block_size,
                       "seq_len_range": [DECODE.len_lo, DECODE.len_hi]},
            "l2": "flushed before every step (512 MiB write, outside the kernel events)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "prefill_ms": round(res["ms_pre"], 5),
        "roofline": {
            "kernel": "attn_fwd_kernel<128>",
            "bound": "tensor",
            "achieved": round(tf_rank, 2),
            "peak": peaks["bf16_tflops"],
            "peak_source": f"{src} dense bf16 (burst)",
            "unit": "TFLOP/s",
            "frac": round(frac, 4),
            "traffic": load_traffic("attn_fwd_kernel<128>"),
            "algorithmic_bytes": PREFILL.io_bytes(),
        },
        "paged_decode": {
            "value": round(gbs, 1),
            "unit": "GB/s",
            "ms": round(res["ms_dec"], 5),
            "kv_bytes": res["kv_bytes"],
            "bytes_per_step": dec_bytes,
            "roofline": {"kernel": "paged_decode_split_kernel<128> + merge", "bound": "hbm",
                         "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "peak_source": f"{src} copy bandwidth", "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": load_traffic("paged_decode_split_kernel<128>")},
        },
        "e2e": {"value": round(e2e_tf, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": round(res["ms_e2e"], 4)},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "wall_s_timed": round(res["wall"], 4),
    }
    if res["cpu"] is not None:
        line["cpu_baseline"] = res["cpu"]
    return line


# --------------------------------------------------------------------------- #
# reference arm: the fp64 oracle on the host cores
# --------------------------------------------------------------------------- #
def run_reference(args):
    qn, kn, vn = synth.prefill_inputs(PREFILL)
    per_step = max(0.5, min(10.0, args.ref_budget_s / max(1, args.steps + args.warmup)))
    tfs = []
    info = None
    for i in range(args.warmup + args.steps):
        tf, info = oracle_prefill_sample(qn, kn, vn, per_step, PREFILL.seed + 1000 + i)
        if i >= args.warmup:
            tfs.append(tf)
    value = statistics.mean(tfs)
    flops = PREFILL.flops()
    return {
        "metric": METRIC,
        "impl": "reference",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": flops / (value * 1e12) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs widened to fp64)",
        "config": {"workload": workload_name(), "note": "each step times the fp64 CPU oracle on "
                   "a bounded random sample of query rows of the prefill workload; ms_per_step "
                   "is the extrapolated time of a full step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": info["cores"],
                         "kind": "oracle",
                         "sample": f"{info['rows']} random query rows per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend="nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(report_ours(args, res, world)), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

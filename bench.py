#!/usr/bin/env python
"""Throughput of the sparse-attention forward (and backward) on GB300.

One step = one `bigbird_attn_fwd` (or `longformer_attn_fwd`) call over the
whole synthetic workload (default: BigBird-ITC, B=8, H=12, n=4096, d=64,
b=64, g=2, w=3, r=3, bf16). The `*_bwd_*` workloads time one
`bigbird_attn_bwd` / `longformer_attn_bwd` call instead (10*d useful FLOPs
per attended pair). Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference|blockified]

Metric: useful TFLOP/s = 4*d * attended (valid query, allowed valid key)
pairs / time. Inputs are resident in HBM before the timed region; L2 is
flushed (256 MiB write) between timed steps, outside the timed events.
`e2e` repeats the measurement through the host-buffer entry point
(`bigbird_attn_fwd_host` / `longformer_attn_fwd_host`) on pinned HOST buffers:
every host->device copy of Q, K, V (and the tables) and the device->host copy
of O is inside the timed region; the library pipelines them against the
computation chunk by chunk. `--impl reference` times the float64 CPU oracle instead.
`--impl blockified` times the pages' own dense-operation formulation in plain
PyTorch on the same GPU (``baselines/blockified.py``: BigBird App. D Eq. (13),
Longformer App. A chunks) on the same inputs and work count; the default line
also carries that baseline's time in `blockified_baseline`.
Multi-GPU (torchrun): every rank runs its own batch of B sequences drawn
from its own seeds, so the global batch is world x B (weak scaling, no
collective on the data path); the step time is the max over ranks.
"""

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

from block_sparse_long_bigbird_gb300.workloads import HEADLINE, WORKLOADS  # noqa: E402

METRIC = "useful TFLOP/s and tokens/s of sparse attn fwd at n=4096, % of bf16 tensor peak"
METRIC_BWD = "useful TFLOP/s and tokens/s of sparse attn bwd (dQ, dK, dV) at n=4096, % of bf16 tensor peak"
UNIT = "TFLOP/s"
# useful FLOPs per attended pair, in units of d: the score (2d) and the P.V
# accumulation (2d) forward; five such products backward
FWD_FLOPS_PER_PAIR_PER_D = 4
BWD_FLOPS_PER_PAIR_PER_D = 10
L2_FLUSH_BYTES = 256 << 20
TC_SOURCE = os.path.join(ROOT, "block_sparse_long_bigbird_gb300", "csrc", "tc_kernel.cuh")
TC_BWD_SOURCE = os.path.join(ROOT, "block_sparse_long_bigbird_gb300", "csrc", "tc_bwd.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference", "blockified"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-blockified", action="store_true", help="skip the dense-formulation baseline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU baseline time budget")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(per_rank_ms, flops_per_rank_step, tokens_per_rank_step):
    """Whole-job throughput: work of all ranks over the slowest rank's step time."""
    world = len(per_rank_ms)
    t = max(per_rank_ms) * 1e-3
    return {
        "ms_per_step": max(per_rank_ms),
        "tflops": world * flops_per_rank_step / t / 1e12,
        "tokens_per_s": world * tokens_per_rank_step / t,
    }


def rank_seed_offset(rank):
    """Seed offset of a rank's own batch: under torchrun the global batch is
    world x B sequences and rank k draws sequences [k B, (k + 1) B) from its
    own seeds (cfg_id + 100 k), so no rank needs another rank's data."""
    return 100 * rank


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def read_traffic(kernel, workload, source=TC_SOURCE):
    """DRAM bytes per launch from a committed ncu capture, if the kernel source is unchanged."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        entries = json.load(f)
    sha = file_sha(source)
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and e.get("source_sha") == sha:
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def make_inputs(wl, rank=0):
    """Seeded synthetic inputs on the CPU (the shared generators only: no
    pattern table and no work count, which each side makes for itself)."""
    import torch

    from block_sparse_long_bigbird_gb300.inputs import make_grad_out, make_key_mask, make_qkv

    Q, K, V = make_qkv(wl.B, wl.H, wl.n, wl.d, wl.dtype, sigma=wl.sigma, cfg_id=wl.cfg_id + rank_seed_offset(rank))
    km = make_key_mask(wl.B, wl.n) if wl.padded else None
    prob = {"Q": Q, "K": K, "V": V, "key_mask": km}
    if wl.grad:
        prob["dO"] = make_grad_out(wl.B, wl.H, wl.n, wl.d, wl.dtype, cfg_id=wl.cfg_id + rank_seed_offset(rank))
    if wl.gproj:
        prob["Qg"], prob["Kg"], prob["Vg"] = make_qkv(wl.B, wl.H, wl.n, wl.d, wl.dtype, sigma=wl.sigma,
                                                      cfg_id=wl.cfg_id + rank_seed_offset(rank) + 1)
    if wl.dilation:
        prob["dilation"] = torch.tensor(wl.dilation, dtype=torch.int32)
    if wl.kind != "bigbird":
        prob["gidx"] = torch.arange(wl.n_global, dtype=torch.int32)
    prob["tokens"] = wl.B * wl.n if km is None else int(km.sum())
    return prob


def make_problem(wl, rank=0):
    """The product side of one step: inputs, the library's pattern table and
    the useful-work count of one step (the library's host accounting)."""
    import block_sparse_long_bigbird_gb300 as sa
    from block_sparse_long_bigbird_gb300 import accounting

    prob = make_inputs(wl, rank)
    km = prob["key_mask"]
    if wl.kind == "bigbird":
        table = sa.build_bigbird_pattern(wl.seed, wl.H, wl.n, wl.b, wl.g, wl.w, wl.r)
        prob["table"] = table
        if km is None:
            pairs = accounting.bigbird_pairs(wl.n, wl.b, wl.g, wl.w, table.numpy()) * wl.B
        else:
            pairs = accounting.bigbird_pairs(wl.n, wl.b, wl.g, wl.w, table.numpy(), km.numpy())
    else:
        dil = wl.dilation or (0,) * wl.H
        pairs = sum(accounting.longformer_pairs(wl.n, wl.window, prob["gidx"].numpy(),
                                                None if km is None else km.numpy(), dilation=dh, causal=wl.causal)
                    for dh in dil)
        if km is None:
            pairs *= wl.B
    prob["pairs"] = pairs
    per_pair = accounting.BWD_FLOPS_PER_PAIR_PER_D if wl.grad else accounting.FWD_FLOPS_PER_PAIR_PER_D
    prob["flops"] = float(per_pair) * wl.d * pairs
    return prob


def call(wl, dev_t, out, stream=None):
    import block_sparse_long_bigbird_gb300 as sa

    if wl.grad:
        if wl.kind == "bigbird":
            sa.bigbird_attn_bwd(dev_t["Q"], dev_t["K"], dev_t["V"], dev_t["dO"], wl.b, wl.g, wl.w, wl.r,
                                dev_t["table"], dev_t.get("key_mask"), out=out, stream=stream)
        else:
            sa.longformer_attn_bwd(dev_t["Q"], dev_t["K"], dev_t["V"], dev_t["dO"], wl.window, dev_t["gidx"],
                                   dev_t.get("key_mask"), out=out, stream=stream)
        return
    if wl.kind == "bigbird":
        sa.bigbird_attn_fwd(dev_t["Q"], dev_t["K"], dev_t["V"], wl.b, wl.g, wl.w, wl.r, dev_t["table"],
                            dev_t.get("key_mask"), out=out, stream=stream)
    else:
        sa.longformer_attn_fwd(dev_t["Q"], dev_t["K"], dev_t["V"], wl.window, dev_t["gidx"],
                               dev_t.get("key_mask"), out=out, stream=stream, dilation=dev_t.get("dilation"),
                               causal=wl.causal, Qg=dev_t.get("Qg"), Kg=dev_t.get("Kg"), Vg=dev_t.get("Vg"))


LONG_SEQ = 8192  # beyond this the CPU baseline samples rows instead of whole heads


def cpu_oracle_sample(wl, prob, budget_s):
    """Time the float64 oracle on the workload until `budget_s` is used: whole
    (batch, head) pairs, or for sequences longer than LONG_SEQ blocks of rows
    of successive heads (credited with the exact pair count of those rows)."""
    import numpy as np

    from oracle import (bigbird_allowed, bigbird_attended_pairs, bigbird_random_table, longformer_allowed,
                        longformer_attended_pairs, masked_attention_grads, oracle_bigbird, oracle_bigbird_bwd,
                        oracle_longformer, oracle_longformer_bwd)

    Q, K, V, km = prob["Q"], prob["K"], prob["V"], prob["key_mask"]
    # The oracle side draws its own pattern table and counts its own work; it
    # takes only the seeded inputs from the shared generators.
    per_pair = float(BWD_FLOPS_PER_PAIR_PER_D if wl.grad else FWD_FLOPS_PER_PAIR_PER_D)
    table = bigbird_random_table(wl.seed, wl.H, wl.n, wl.b, wl.g, wl.w, wl.r) if wl.kind == "bigbird" else None
    heads = [(beta, h) for beta in range(wl.B) for h in range(wl.H)]
    long_seq = wl.n > LONG_SEQ
    nrows = max(64, min(1024, (1 << 24) // wl.n))  # the dense masked oracle costs n per row
    rows = np.arange(wl.n // 2, wl.n // 2 + nrows) if long_seq else None  # a block of rows mid-sequence
    done, flops = 0, 0.0
    t0 = time.perf_counter()
    for beta, h in heads:
        sl = (slice(beta, beta + 1), slice(h, h + 1))
        kmb = None if km is None else km[beta:beta + 1].numpy()
        kv = None if kmb is None else kmb[0] != 0
        if wl.kind == "bigbird":
            tab = table[h:h + 1]
            if long_seq:
                mask = bigbird_allowed(wl.n, wl.b, wl.g, wl.w, tab[0], rows)
                if kv is not None:
                    mask = mask & kv[None, :] & kv[rows][:, None]
                if wl.grad:
                    # every backward product for the row block's pairs: its dQ rows and
                    # its contributions to dK and dV
                    masked_attention_grads(Q[beta, h, rows], K[beta, h], V[beta, h], mask, prob["dO"][beta, h, rows])
                else:
                    oracle_bigbird(Q[sl], K[sl], V[sl], wl.b, wl.g, wl.w, tab, key_mask=kmb, rows=rows)
            elif wl.grad:
                oracle_bigbird_bwd(Q[sl], K[sl], V[sl], prob["dO"][sl], wl.b, wl.g, wl.w, tab, key_mask=kmb)
            else:
                oracle_bigbird(Q[sl], K[sl], V[sl], wl.b, wl.g, wl.w, tab, key_mask=kmb)
            if long_seq:
                flops += per_pair * wl.d * int(mask.sum())
            else:
                flops += per_pair * wl.d * bigbird_attended_pairs(wl.n, wl.b, wl.g, wl.w, tab, key_mask=kmb)
        else:
            gi = prob["gidx"].numpy()
            dh = wl.dilation[h] if wl.dilation else 0
            gsl = {k: prob[k][sl] for k in ("Qg", "Kg", "Vg")} if wl.gproj else {}
            if wl.grad:
                oracle_longformer_bwd(Q[sl], K[sl], V[sl], prob["dO"][sl], wl.window, gi, key_mask=kmb,
                                      dilation=[dh], causal=wl.causal, **gsl)
                flops += per_pair * wl.d * longformer_attended_pairs(wl.n, wl.window, gi, key_mask=kmb,
                                                                     dilation=[dh], causal=wl.causal)
            else:
                oracle_longformer(Q[sl], K[sl], V[sl], wl.window, gi, key_mask=kmb, rows=rows, dilation=[dh],
                                  causal=wl.causal, **gsl)
                if long_seq:
                    mask = longformer_allowed(wl.n, wl.window, gi, rows, dilation=dh, causal=wl.causal)
                    if kv is not None:
                        mask = mask & kv[None, :] & kv[rows][:, None]
                    flops += per_pair * wl.d * int(mask.sum())
                else:
                    flops += per_pair * wl.d * longformer_attended_pairs(wl.n, wl.window, gi, key_mask=kmb,
                                                                         dilation=[dh], causal=wl.causal)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info

        cores = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        cores = len(os.sched_getaffinity(0))
    what = (f"rows [n/2, n/2 + {nrows}) (dense masked float64, all n keys per row; backward: every product "
            f"of those rows' pairs) of") if long_seq else "all rows of"
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{what} {done} of {len(heads)} (batch, head) pairs, float64 numpy, {dt:.1f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    prob = make_inputs(wl)  # the oracle arm loads no product code
    budget = max(0.5, min(args.cpu_seconds, 120.0) / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, prob, 0.0)
    vals, times = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        r = cpu_oracle_sample(wl, prob, budget)
        times.append(time.perf_counter() - t0)
        vals.append(r["value"])
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC_BWD if wl.grad else METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": "per step: " + r["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def blockified_unsupported(wl):
    """Why the dense-formulation baseline cannot run `wl`, or None."""
    if wl.grad:
        return "the pages give the dense formulation for the forward only"
    if wl.kind == "longformer" and (wl.dilation and any(wl.dilation)):
        return "the chunks formulation (Longformer App. A) supports only the non-dilated window"
    if wl.gproj:
        return "the chunks formulation has no separate global projections"
    return None


def blockified_call(wl, dev_t):
    from baselines.blockified import bigbird_blockified, longformer_chunks

    if wl.kind == "bigbird":
        return bigbird_blockified(dev_t["Q"], dev_t["K"], dev_t["V"], wl.b, wl.g, wl.w, wl.r, dev_t.get("table"),
                                  dev_t.get("key_mask"))
    return longformer_chunks(dev_t["Q"], dev_t["K"], dev_t["V"], wl.window, dev_t["gidx"], dev_t.get("key_mask"),
                             causal=wl.causal)


def time_blockified(wl, dev_t, flush, stream, steps, warmup):
    """CUDA-event time of the dense-formulation baseline, same protocol as the
    library's timed steps (L2 flushed between steps, outside the events)."""
    import torch

    for _ in range(max(3, warmup)):
        blockified_call(wl, dev_t)
    torch.cuda.synchronize()
    ms = []
    for i in range(steps):
        flush.fill_(i & 0xFF)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        blockified_call(wl, dev_t)
        e.record(stream)
        torch.cuda.synchronize()
        ms.append(s.elapsed_time(e))
    return ms


def run_blockified(args):
    """The pages' dense formulation on this GPU, as its own bench line."""
    import torch

    rank, world, local = dist_env()
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    why = blockified_unsupported(wl)
    if why:
        print(json.dumps({"impl": "blockified", "unavailable": why}), flush=True)
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    prob = make_problem(wl)
    dev_t = {k: v.to(dev) for k, v in prob.items() if hasattr(v, "to") and v is not None}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    with ClockSampler(local) as clocks:
        ms = time_blockified(wl, dev_t, flush, stream, args.steps, args.warmup)
    t = sum(ms) / len(ms)
    # end to end: pinned host inputs copied in, the dense formulation, the output copied back
    ins = [k for k in ("Q", "K", "V", "table", "gidx", "key_mask") if prob.get(k) is not None]
    host = {k: prob[k].pin_memory() for k in ins}
    O = blockified_call(wl, dev_t)
    out_h = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    e_ms = []
    for i in range(max(2, args.warmup) + args.steps):
        flush.fill_(i & 0xFF)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for k in ins:
            dev_t[k].copy_(host[k], non_blocking=True)
        out_h.copy_(blockified_call(wl, dev_t), non_blocking=True)
        e.record(stream)
        torch.cuda.synchronize(dev)
        if i >= max(2, args.warmup):
            e_ms.append(s.elapsed_time(e))
    e_t = sum(e_ms) / len(e_ms)
    peaks, peak_src = read_peaks()
    value = prob["flops"] / (t * 1e-3) / 1e12
    line = {
        "impl": "blockified", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": t, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded torch.randn inputs, pattern seed 0)", "config": workload_config(wl),
        "frac_of_bf16_peak": value / peaks["bf16_tflops"],
        "e2e": {"value": prob["flops"] / (e_t * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": e_t,
                "h2d_bytes_per_step": sum(host[k].numel() * host[k].element_size() for k in ins),
                "d2h_bytes_per_step": out_h.numel() * out_h.element_size()},
        "clocks": clocks.summary(), "per_step_ms": {"min": min(ms), "median": statistics.median(ms), "max": max(ms)},
        "note": "plain PyTorch dense operations (cuBLAS batched products, fp32 softmax); useful FLOPs as for "
                "the library: 4*d per attended pair",
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl):
    cfg = {"workload": f"{wl.name}: {wl.kind}{' backward' if wl.grad else ''} B={wl.B} H={wl.H} n={wl.n} d={wl.d}",
           "B": wl.B, "H": wl.H, "n": wl.n, "d": wl.d, "dtype": wl.dtype,
           "l2": "flushed between timed steps (256 MiB write), inputs resident in HBM"}
    if wl.kind == "bigbird":
        cfg.update({"b": wl.b, "g": wl.g, "w": wl.w, "r": wl.r, "pattern_seed": wl.seed})
    else:
        cfg.update({"window": wl.window, "n_global": wl.n_global})
        if wl.dilation:
            cfg["dilation"] = list(wl.dilation)
        if wl.causal:
            cfg["causal"] = True
        if wl.gproj:
            cfg["separate_global_projections"] = True
    if wl.padded:
        cfg["key_padding"] = "lengths ~ U[n/2, n] (seed 2000)"
    return cfg


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.impl == "blockified":
        return run_blockified(args)

    import torch

    import block_sparse_long_bigbird_gb300 as sa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[args.workload]
    prob = make_problem(wl, rank)
    dev_t = {k: v.to(dev) for k, v in prob.items() if hasattr(v, "to") and v is not None}
    out = tuple(torch.empty_like(dev_t["Q"]) for _ in range(3)) if wl.grad else torch.empty_like(dev_t["Q"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        call(wl, dev_t, out)
    torch.cuda.synchronize(dev)
    status = sa.get_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after warm-up: {status}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    gpu_id = local
    try:
        gpu_id = torch.cuda.get_device_properties(dev).uuid
        gpu_id = "GPU-" + str(gpu_id) if not str(gpu_id).startswith("GPU-") else str(gpu_id)
    except Exception:
        pass
    barrier()
    launches = 0
    with ClockSampler(gpu_id) as clocks:
        # the sampler's start-up pause idles the GPU; two more untimed calls
        # bring the clocks back up before the first timed step
        for _ in range(2):
            call(wl, dev_t, out)
        barrier()
        # one more untimed call, not waited for, so that the device is busy when
        # the first timed step's start event is recorded (otherwise the host's
        # time to enqueue that step's kernel after an idle device is counted)
        flush.fill_(0xFF)
        call(wl, dev_t, out)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            call(wl, dev_t, out)
            ends[i].record(stream)
            launches += sa.last_launch_count()
        barrier()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    my_ms = sum(ms) / len(ms)
    if world > 1:
        import torch.distributed as dist

        t = torch.tensor([my_ms], dtype=torch.float64, device=dev)
        gathered = [torch.zeros_like(t) for _ in range(world)]
        dist.all_gather(gathered, t)
        per_rank = [float(x.item()) for x in gathered]
    else:
        per_rank = [my_ms]
    agg = aggregate(per_rank, prob["flops"], prob["tokens"])
    status = sa.get_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status after timed steps: {status}")

    peaks, peak_src = read_peaks()
    kernel_tflops = prob["flops"] / (my_ms * 1e-3) / 1e12
    kernel_name = "sparse_tc_fwd<{},{},{}>".format(wl.d, "padded" if wl.padded else "dense",
                                                   "longformer" if wl.kind == "longformer" else "bigbird")
    if wl.grad:
        # one call launches the row pass and the key pass; they are timed together
        kernel_name = f"sparse_tc_bwd<{wl.d},rows> + sparse_tc_bwd<{wl.d},keys>"
    traffic = read_traffic(kernel_name, wl.name, TC_BWD_SOURCE if wl.grad else TC_SOURCE)
    roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": kernel_tflops / peaks["bf16_tflops"], "traffic": traffic,
                "peak_source": f"{peak_src} bf16 dense burst (cuBLAS)", "kernel": kernel_name,
                "algorithmic_flops_per_launch": prob["flops"]}
    hbm_bytes = (8 if wl.grad else 4) * wl.B * wl.H * wl.n * wl.d * (2 if wl.dtype == "bf16" else 4)
    roofline["hbm_frac_of_min_bytes"] = hbm_bytes / (my_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]

    e2e = None
    if not args.no_e2e:
        if wl.grad or wl.gproj:
            # backward (and the separate-projection forward, which has no
            # host-buffer entry point): host->device copies of the inputs, the
            # device call, device->host copies of the outputs, all on the
            # launching stream
            ins = ("Q", "K", "V", "dO") if wl.grad else ("Q", "K", "V", "Qg", "Kg", "Vg")
            outs = out if wl.grad else (out,)
            host = {k: prob[k].pin_memory() for k in ins}
            out_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]

            def e2e_step():
                for k in ins:
                    dev_t[k].copy_(host[k], non_blocking=True)
                call(wl, dev_t, out)
                for oh, o in zip(out_h, outs):
                    oh.copy_(o, non_blocking=True)

            h2d = sum(prob[k].numel() * prob[k].element_size() for k in ins)
            d2h = sum(o.numel() * o.element_size() for o in outs)
        else:
            # forward: the host-buffer entry point, which pipelines the copies
            # against the computation chunk by chunk
            host = {k: prob[k].pin_memory() for k in ("Q", "K", "V")}
            tabs = {k: prob[k] for k in ("table", "gidx", "key_mask", "dilation") if prob.get(k) is not None}
            out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()

            def e2e_step():
                if wl.kind == "bigbird":
                    sa.bigbird_attn_fwd_host(host["Q"], host["K"], host["V"], wl.b, wl.g, wl.w, wl.r,
                                             tabs.get("table"), tabs.get("key_mask"), out=out_h, stream=stream)
                else:
                    sa.longformer_attn_fwd_host(host["Q"], host["K"], host["V"], wl.window, tabs.get("gidx"),
                                                tabs.get("key_mask"), out=out_h, stream=stream,
                                                dilation=tabs.get("dilation"), causal=wl.causal)

            h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + list(tabs.values()))
            d2h = out_h.numel() * out_h.element_size()
        e_ms = []
        for i in range(max(2, args.warmup) + args.steps):
            flush.fill_(i & 0xFF)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            e2e_step()
            e.record(stream)
            torch.cuda.synchronize(dev)
            if i >= max(2, args.warmup):
                e_ms.append(s.elapsed_time(e))
        e_t = sum(e_ms) / len(e_ms)
        if world > 1:
            import torch.distributed as dist

            t = torch.tensor([e_t], dtype=torch.float64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e_t = float(t.item())
        e2e = {"value": world * prob["flops"] / (e_t * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": e_t, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "api": "device call with stream-ordered copies" if (wl.grad or wl.gproj)
               else f"{wl.kind}_attn_fwd_host (host buffers, copies pipelined in the library)"}

    blk = None
    if rank == 0 and world == 1 and not args.no_blockified:
        why = blockified_unsupported(wl)
        if why:
            blk = {"unavailable": why}
        else:
            try:
                b_ms = time_blockified(wl, dev_t, flush, stream, args.steps, args.warmup)
                b_t = sum(b_ms) / len(b_ms)
                blk = {"value": prob["flops"] / (b_t * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": b_t,
                       "what": "the pages' dense formulation in plain PyTorch on this GPU, same inputs "
                               "(baselines/blockified.py)"}
            except torch.cuda.OutOfMemoryError as exc:
                blk = {"unavailable": f"out of memory: {str(exc).splitlines()[0]}"}
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(wl, prob, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC_BWD if wl.grad else METRIC, "value": agg["tflops"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": agg["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic (seeded torch.randn inputs, pattern seed 0)",
            "config": workload_config(wl),
            "tokens_per_s": agg["tokens_per_s"],
            "useful_gflop_per_step": prob["flops"] / 1e9,
            "frac_of_bf16_peak": agg["tflops"] / world / peaks["bf16_tflops"],
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "blockified_baseline": blk,
            "gpu_launches": launches, "clocks": clocks.summary(),
            "per_step_ms": {"min": min(ms), "median": statistics.median(ms), "max": max(ms)},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the hot path: BlockMask creation + block-sparse masked attention forward (and the paged
split-KV decode as a secondary line item), on seeded synthetic inputs, through the C ABI.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload cfg2|cfg3|cfg4]

A step = fa_create_block_mask + fa_flex_forward over the whole workload (default: plain causal, B=4,
Hq=Hkv=16, N=4096, d=128, 128x128 blocks). value = physical TFLOP/s (4*d*Bq*Bk per visited block per
(b,h)) of the whole step, all ranks. The other prefill workloads (document-causal + ALiBi N=16384; sliding
window 1024 + soft-cap N=65536) are timed the same way and reported as objects of the same line, beside
the paged decode, the backward and the paged prefill. One JSON line on rank 0.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-sparse attn fwd TFLOP/s (% BF16 tc peak); decode KV GB/s (% HBM)"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="cfg2", choices=["cfg2", "cfg3", "cfg4"])
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--decode-only", action="store_true",
                   help="time only the paged decode and print its object as the line (profiling aid)")
    p.add_argument("--decode-requests", type=int, default=64, help="requests in the decode batch")
    p.add_argument("--no-backward", action="store_true")
    p.add_argument("--no-paged", action="store_true")
    p.add_argument("--no-others", action="store_true", help="skip the other prefill workloads")
    p.add_argument("--no-split", action="store_true", help="skip the split-row prefill line")
    p.add_argument("--backward-only", action="store_true",
                   help="after the forward, time only the backward and print its object as the line (profiling aid)")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return dict(hbm=float(m["hbm_gbs"]), bf16=float(m["bf16_tflops"]),
                    bf16_sus=float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def make_workload(name):
    from block_sparse_masked_create_gb300 import workloads
    return {"cfg2": workloads.cfg2, "cfg3": workloads.cfg3, "cfg4": workloads.cfg4}[name]()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.samples = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append([x.strip() for x in line.split(",")])

    def busy_until_sampled(self, work, n=3, max_s=8.0):
        """Run `work` (GPU work + sync) until the sampler has seen n samples, so that the timed region
        that follows sits inside a sampled window under the same load."""
        t0 = time.perf_counter()
        while self.proc and len(self.samples) < n and time.perf_counter() - t0 < max_s:
            work()

    def busy_for(self, work, seconds):
        t0 = time.perf_counter()
        while self.proc and time.perf_counter() - t0 < seconds:
            work()

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            try:
                sm.append(float(s[1]))
                mx = float(s[2])
                for n, v in zip(names, s[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
            except Exception:
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "window": "200 ms samples while the step runs back to back, before, during "
                                              "and after the timed region"}


# ------------------------------------------------------------------------------------------------------
# reference arm / CPU baseline: the fp64 oracle as it stands, on a bounded sample, on host cores
# ------------------------------------------------------------------------------------------------------
CPU_SNIPPET = r"""
import json, sys, time, numpy as np
sys.path.insert(0, %(root)r)
from block_sparse_masked_create_gb300 import workloads, synth
from oracle import flexmask_oracle as orc
w = workloads.%(wl)s()
rng = np.random.default_rng(%(seed)d)
g = w.Hq // w.Hkv
n_q = -(-w.q_len // w.bq)
score = {k: (np.asarray(v, np.float64) if k != 'softcap' else v) for k, v in w.score.items()}
times, flops = [], []
while len(times) < %(reps)d and sum(times) < %(seconds)f:
    b, h, r = int(rng.integers(w.B)), int(rng.integers(w.Hq)), int(rng.integers(n_q))
    rows = np.arange(r * w.bq, min(w.q_len, (r + 1) * w.bq))
    hk = h // g
    # inputs of this sample only (generator slices: counter based)
    qb = synth.normal_bf16_bits(w.seed, 1, (len(rows), w.d), first=((b * w.Hq + h) * w.q_len + rows[0]) * w.d)
    kb = synth.normal_bf16_bits(w.seed, 2, (w.kv_len, w.d), first=(b * w.Hkv + hk) * w.kv_len * w.d)
    vb = synth.normal_bf16_bits(w.seed, 3, (w.kv_len, w.d), first=(b * w.Hkv + hk) * w.kv_len * w.d)
    qf, kf, vf = (synth.bf16_bits_to_f64(x) for x in (qb, kb, vb))
    t = orc.block_mask(w.rule, 1, 1, w.q_len, w.kv_len, w.bq, w.bk, doc_ids=w.doc_ids, rows=[r])
    vis = int(t["kv_num"][0, 0, r] + t["full_kv_num"][0, 0, r])
    t0 = time.perf_counter()
    orc.attention_rows(qf, kf, vf, w.rule, rows, b, h, w.q_len, w.kv_len, w.scale, score, 0, w.doc_ids)
    times.append(time.perf_counter() - t0)
    flops.append(4.0 * w.d * w.bq * w.bk * vis)
print(json.dumps({"times": times, "flops": flops}))
"""


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_oracle_parallel(wl: str, reps: int, seconds: float, workers: int) -> dict:
    """The oracle as it stands on `workers` host cores: one single-threaded worker process per core, each
    timing the oracle on its own seeded sample of query-block rows (at most `reps` rows or `seconds` of
    oracle time). The processes are started with exec (no fork of a CUDA context)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    procs = [subprocess.Popen([sys.executable, "-c", CPU_SNIPPET % dict(root=ROOT, wl=wl, reps=reps,
                                                                        seconds=seconds, seed=i)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env)
             for i in range(workers)]
    res = []
    for p in procs:
        out, err = p.communicate(timeout=1800)
        if p.returncode != 0:
            raise RuntimeError(err[-2000:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    return {"workers": res}


def max_over_ranks(ms: float, dist=None, device=None) -> float:
    """The job's time is the slowest rank's: all-reduce MAX of each rank's timed region (ms)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist=None, device=None) -> float:
    """The job's work: all-reduce SUM of each rank's own work (every unit belongs to one rank)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_tflops(world: int, flop_per_rank: float, ms_step: float) -> float:
    """Whole-job throughput: every rank processes its own shard of flop_per_rank per step (weak scaling)."""
    return world * flop_per_rank / (ms_step * 1e-3) / 1e12


def reference_arm(args, rank):
    if rank != 0:
        return
    w = make_workload(args.workload)
    cores = host_cores()
    # a step = one query-block row of a random (b, h) on every host core, in parallel
    res = run_oracle_parallel(args.workload, args.warmup + args.steps, 1e9, cores)["workers"]
    t_w = [sum(r["times"][args.warmup:]) for r in res]
    f_tot = sum(sum(r["flops"][args.warmup:]) for r in res)
    value = f_tot / max(t_w) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * max(t_w) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} N={w.q_len} d={w.d} Bq=Bk={w.bq}",
                   "step": f"oracle on one query block row (Bq rows) of a random (b, h) per host core, {cores} cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} timed query-block rows of {w.bq} queries per core "
                                   f"(fp64 numpy, one single-threaded process per core)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------------
LOGICAL_NOTE = "valid (query, key) pairs from the rule's closed form"


def logical_pairs_of(name, w):
    """Exact count of allowed (query, key) pairs of a prefill workload, from closed forms of its rule
    (causal: n(n+1)/2 per head; window W: W(W+1)/2 + (n-W)W; document-causal: sum of len(len+1)/2)."""
    if name == "cfg2":
        return w.B * w.Hq * w.q_len * (w.q_len + 1) // 2
    if name == "cfg4":
        W = 1024
        return w.B * w.Hq * (W * (W + 1) // 2 + (w.q_len - W) * W)
    if name == "cfg3":
        return w.B * w.Hq * int(sum(int(L) * (int(L) + 1) // 2 for L in w.doc_lens))
    return None


class Prefill:
    """One prefill workload resident on the device: inputs, rule, BlockMask, outputs (fp32 O, as the
    tolerance needs), and the work counts of its visited blocks."""

    def __init__(self, name, dev, w=None):
        import numpy as np
        import torch

        from block_sparse_masked_create_gb300 import fa, workloads
        self.name = name
        w = self.w = make_workload(name).generate() if w is None else w
        self.q = workloads.bf16_torch(w.q_bits, dev)
        self.k = workloads.bf16_torch(w.k_bits, dev)
        self.v = workloads.bf16_torch(w.v_bits, dev)
        self.doc = None if w.doc_ids is None else torch.from_numpy(w.doc_ids.astype(np.int32)).to(dev)
        al = None
        if w.score.get("alibi_slopes") is not None:
            al = torch.tensor(np.asarray(w.score["alibi_slopes"], np.float32), device=dev)
        self.al = al
        self.sc = fa.make_score_rule(al, None, w.score.get("softcap", 0.0))
        self.rule = fa.make_mask_rule(w.rule, doc_ids=self.doc)
        self.bm = fa.create_block_mask(self.rule, w.B, w.Hq, w.q_len, w.kv_len, w.bq, w.bk, device=dev,
                                       keep=[self.doc])
        self.out = torch.empty(self.q.shape, dtype=torch.float32, device=dev)
        self.lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stats = fa.block_mask_stats(self.bm).cpu().tolist()
        heads = w.B * w.Hq // (self.bm.c.Bm * self.bm.c.Hm)
        self.visited = (self.stats[0] + self.stats[1]) * heads
        self.phys_flops = 4.0 * w.d * w.bq * w.bk * self.visited
        self.logical_pairs = logical_pairs_of(name, w)
        self.launches = 3 + (1 if w.doc_ids is not None else 0)   # doc runs, classify, transpose, forward

    def mask(self):
        from block_sparse_masked_create_gb300 import fa
        w = self.w
        fa.recreate_block_mask(self.bm, self.rule, w.B, w.Hq, w.q_len, w.kv_len, w.bq, w.bk)

    def forward(self):
        from block_sparse_masked_create_gb300 import fa
        fa.flex_forward(self.q, self.k, self.v, self.bm, self.sc, self.w.scale, out=self.out, lse=self.lse,
                        status=self.status)

    def step(self):
        self.mask()
        self.forward()

    def row_lengths(self):
        """Visited blocks (full + partial) per query block row of the table: mean, P50, P95, max ([FX] 5:
        row lengths as the load signal)."""
        import numpy as np
        t = self.bm.tables()
        ln = (t["kv_num"] + t["full_kv_num"]).flatten().cpu().numpy().astype(np.float64)
        return {"mean": float(ln.mean()), "p50": float(np.percentile(ln, 50)), "p95": float(np.percentile(ln, 95)),
                "max": int(ln.max()), "rows": int(ln.size), "nk": int(self.bm.c.nk)}

    def config(self):
        w = self.w
        return f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} N={w.q_len} d={w.d} Bq=Bk={w.bq}"


class Shard:
    """One rank's share of a workload partitioned by (batch row, KV head) units: its pieces (each a local
    problem with its own mask), run one after the other; the same interface as Prefill."""

    def __init__(self, name, parts, desc):
        self.name, self.parts, self.desc = name, parts, desc
        self.w = parts[0].w
        self.phys_flops = sum(p.phys_flops for p in parts)
        self.visited = sum(p.visited for p in parts)
        lp = [p.logical_pairs for p in parts]
        self.logical_pairs = None if any(x is None for x in lp) else sum(lp)
        self.stats = [sum(p.stats[i] for p in parts) for i in range(3)] + [max(p.stats[3] for p in parts)]
        self.launches = sum(p.launches for p in parts)
        self.status = parts[0].status

    def mask(self):
        for p in self.parts:
            p.mask()

    def forward(self):
        for p in self.parts:
            p.forward()

    def step(self):
        self.mask()
        self.forward()

    def row_lengths(self):
        import numpy as np
        ln = []
        for p in self.parts:
            t = p.bm.tables()
            ln.append((t["kv_num"] + t["full_kv_num"]).flatten().cpu().numpy().astype(np.float64))
        ln = np.concatenate(ln)
        return {"mean": float(ln.mean()), "p50": float(np.percentile(ln, 50)), "p95": float(np.percentile(ln, 95)),
                "max": int(ln.max()), "rows": int(ln.size), "nk": int(self.parts[0].bm.c.nk)}

    def config(self):
        return self.desc


def timed_steps(pf, steps, stream):
    """Per step: events around the mask build and the forward on the launching stream."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        pf.mask()
        ev[i][1].record(stream)
        pf.forward()
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    return (start.elapsed_time(end), [a.elapsed_time(c) for (_, a, c) in ev],
            [s_.elapsed_time(a) for (s_, a, _) in ev])


def prefill_summary(pf, pk, fwd_ms, mask_ms, ms_step, world):
    """The per-workload fields: physical and logical TFLOP/s, the forward's roofline, rho_tile, blocks and
    row lengths."""
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    achieved = pf.phys_flops / (fwd_avg * 1e-3) / 1e12
    logical = pf.logical_pairs
    return {
        "workload": pf.config(),
        "physical_tflop_per_step": pf.phys_flops / 1e12,
        "step_tflops": world * pf.phys_flops / (ms_step * 1e-3) / 1e12,
        "logical_tflops": (world * 4.0 * pf.w.d * logical / (ms_step * 1e-3) / 1e12) if logical else None,
        "logical_pairs_note": LOGICAL_NOTE,
        "rho_tile": (pf.phys_flops / (4.0 * pf.w.d * logical)) if logical else None,
        "pct_bf16_peak": achieved / pk["bf16"],
        "mask_build_us": 1e3 * statistics.median(mask_ms),
        "forward_ms_median": statistics.median(fwd_ms),
        "forward_ms_mean": fwd_avg,
        "blocks": {"full": pf.stats[0], "partial": pf.stats[1], "empty": pf.stats[2], "row_max": pf.stats[3],
                   "visited_total": pf.visited},
        "row_length": pf.row_lengths(),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": achieved / pk["bf16"], "traffic": load_traffic(pf.name),
                     "kernel": "fa_flex_forward", "peak_src": f"{pk['src']} bf16 burst"},
    }


def other_prefill(name, args, dev, pk, world):
    """Another prefill workload timed the same way as the main one (mask build + forward per step)."""
    import torch

    from block_sparse_masked_create_gb300 import fa
    pf = Prefill(name, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        pf.step()
    torch.cuda.synchronize()
    ms, fwd_ms, mask_ms = timed_steps(pf, args.steps, stream)
    o = prefill_summary(pf, pk, fwd_ms, mask_ms, ms / args.steps, world)
    o["ms_per_step"] = ms / args.steps
    o["status"] = fa.status_string(fa.check_status(pf.status))
    o["gpu_launches"] = args.steps * pf.launches
    return o


def copy_ceiling(hq, hk, hv, ho, hl, q, k, v, out, lse, dev):
    """Plain pinned copies of the e2e step's bytes on their own: all inputs host -> device, all outputs
    device -> host, and both directions at once on two streams (the floor for any overlap of the two)."""
    import torch
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)

    def h2d():
        with torch.cuda.stream(s_in):
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            ho.copy_(out, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

    def timed(fns, n=5):
        ms = []
        for it in range(n + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            for st in (s_in, s_out):
                st.wait_event(a)
            for f in fns:
                f()
            for st in (s_in, s_out):
                e = torch.cuda.Event()
                e.record(st)
                main.wait_event(e)
            b.record(main)
            torch.cuda.synchronize()
            if it >= 2:
                ms.append(a.elapsed_time(b))
        return statistics.median(ms)

    bi = (q.numel() + k.numel() + v.numel()) * 2
    bo = out.numel() * out.element_size() + lse.numel() * 4
    t_in, t_out, t_both = timed([h2d]), timed([d2h]), timed([h2d, d2h])
    return {"h2d_ms": t_in, "d2h_ms": t_out, "duplex_ms": t_both, "h2d_GBps": bi / (t_in * 1e-3) / 1e9,
            "d2h_GBps": bo / (t_out * 1e-3) / 1e9,
            "note": "pinned host <-> device copies of the step's input and output bytes alone (CUDA events)"}


def ours(args, rank, world, local_rank):
    import torch

    from block_sparse_masked_create_gb300 import fa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk = peaks()
    if world > 1:
        # the workload with its batch scaled by the number of ranks, partitioned by (batch row, KV head)
        # units: each rank builds masks for and runs only its own units (weak scaling, no collective)
        from block_sparse_masked_create_gb300 import partition
        wg = make_workload(args.workload)
        wg.B *= world
        pieces = partition.pieces_for_rank(wg.B, wg.Hkv, world, rank)
        parts = [Prefill(args.workload, dev, w=partition.slice_prefill(wg, pc)[0]) for pc in pieces]
        pf = Shard(args.workload, parts, pf_config(wg) + f", rank {rank} of {world}: (b, h_kv) pieces {pieces}")
    else:
        pf = Prefill(args.workload, dev)
        parts = [pf]
    w, status = pf.w, pf.status
    phys_flops = pf.phys_flops
    step_launches = pf.launches  # per piece: [document runs,] classify, transpose, forward
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        pf.step()
    torch.cuda.synchronize()
    if fa.check_status(status) != fa.OK:
        raise RuntimeError("device status after warm-up")
    if dist:
        dist.barrier()
    torch.cuda.synchronize()

    def busy():
        for _ in range(20):
            pf.step()
        torch.cuda.synchronize()

    with ClockSampler(local_rank) as clk:
        clk.busy_until_sampled(busy)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        # per-kernel time of the dominant kernel (the forward) with events on the launching stream
        ms, fwd_ms, mask_ms = timed_steps(pf, args.steps, stream)
        wall = time.perf_counter() - t0
        clk.busy_for(busy, 0.5)
    if dist:
        dist.barrier()
    ms = max_over_ranks(ms, dist, dev)
    total_flops = sum_over_ranks(phys_flops, dist, dev)   # every unit counted once, on the rank that owns it
    st_code = fa.check_status(status)
    ms_step = ms / args.steps
    value = total_flops / (ms_step * 1e-3) / 1e12
    summ = prefill_summary(pf, pk, fwd_ms, mask_ms, ms_step, world)

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if rank == 0 or world > 1:
        hosts = []
        for p in parts:
            hq = torch.empty(p.q.shape, dtype=torch.bfloat16, pin_memory=True).copy_(p.q)
            hk = torch.empty(p.k.shape, dtype=torch.bfloat16, pin_memory=True).copy_(p.k)
            hv = torch.empty(p.v.shape, dtype=torch.bfloat16, pin_memory=True).copy_(p.v)
            ho = torch.empty(p.out.shape, dtype=p.out.dtype, pin_memory=True)
            hl = torch.empty(p.lse.shape, dtype=torch.float32, pin_memory=True)
            pw = p.w
            hws = torch.empty(fa.forward_host_workspace_bytes(pw.B, pw.Hq, pw.Hkv, pw.q_len, pw.kv_len, pw.d,
                                                              p.out.dtype), dtype=torch.uint8, device=dev)
            hosts.append((p, hq, hk, hv, ho, hl, hws))

        def e2e_step():  # host tensors in and out: fa_flex_forward_host streams them through the GPU
            for (p, hq, hk, hv, ho, hl, hws) in hosts:
                p.mask()
                fa.flex_forward_host(hq, hk, hv, p.bm, p.sc, p.w.scale, out=ho, lse=hl, workspace=hws,
                                     status=p.status)

        for _ in range(max(3, args.warmup // 2)):
            e2e_step()
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n2 = max(3, args.steps // 2)
        s2.record(stream)
        for _ in range(n2):
            e2e_step()
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2) / n2, dist, dev)
        bi = sum(3 * p.q.numel() * 2 for p in parts)
        bo = sum(p.out.numel() * p.out.element_size() + p.lse.numel() * 4 for p in parts)
        e2e = {"value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms,
               "api": "fa_flex_forward_host (pinned host Q, K, V, O, LSE)"}
        if world == 1:
            (_, hq, hk, hv, ho, hl, _) = hosts[0]
            ceil = copy_ceiling(hq, hk, hv, ho, hl, pf.q, pf.k, pf.v, pf.out, pf.lse, dev)
            e2e.update({"copy_ceiling": ceil, "copy_floor_over_e2e": ceil["duplex_ms"] / e2e_ms})
        del hosts

    # the measurements below are of one GPU: they run with a single rank only
    if world > 1:
        args.no_backward = args.no_paged = args.no_others = args.no_split = args.no_decode = True
        args.no_cpu = True
    else:
        w, q, k, v, out, lse, bm, sc = pf.w, pf.q, pf.k, pf.v, pf.out, pf.lse, pf.bm, pf.sc

    # ---------------- backward over the same mask and forward outputs (secondary line item)
    bwd_line = None
    if not args.no_backward:
        bwd_line = bench_backward(args, dev, pk, w, q, k, v, bm, sc, out, lse, phys_flops)
        if args.backward_only:
            if rank == 0:
                print(json.dumps(bwd_line), flush=True)
            return

    # ---------------- paged prefill: the same forward with K/V behind a page table
    paged_line = None
    if not args.no_paged:
        paged_line = bench_paged_prefill(args, dev, pk, w, q, bm, sc, phys_flops)

    # ---------------- the other prefill workloads, each timed like the main one
    others = {}
    if not args.no_others:
        del pf, parts, q, k, v, out, lse
        torch.cuda.empty_cache()
        for name in ("cfg2", "cfg3", "cfg4"):
            if name != args.workload:
                others[name] = other_prefill(name, args, dev, pk, world)
                torch.cuda.empty_cache()

    # ---------------- split rows: a chunked prefill over a long context, with and without splitting its rows
    split_line = None
    if not args.no_split:
        split_line = bench_split_prefill(args, dev, pk)
        torch.cuda.empty_cache()

    # ---------------- decode (secondary metric of the same hot path): paged split-KV, 64 requests
    dec_line = None
    if not args.no_decode:
        dec_line = bench_decode(args, dev, pk)

    cpu = None
    if rank == 0 and not args.no_cpu:
        cores = host_cores()
        budget = 20.0
        try:
            res = run_oracle_parallel(args.workload, 10 ** 6, max(1.0, budget / cores), cores)["workers"]
            t_w = [sum(r["times"]) for r in res]
            n_rows = sum(len(r["times"]) for r in res)
            cpu = {"value": sum(sum(r["flops"]) for r in res) / max(t_w) / 1e12, "unit": "TFLOP/s",
                   "cores": cores, "kind": "oracle",
                   "sample": f"{n_rows} query-block rows ({w.bq} queries each) of random (b, h) of {w.name}, "
                             f"fp64 numpy, {cores} single-threaded processes, {sum(t_w):.1f} s of oracle time "
                             f"({max(t_w):.1f} s wall per core)"}
        except Exception as e:  # reported, never silently replaced
            cpu = {"value": None, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": f"failed: {e}"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": pf_config(w) if world == 1 else summ["workload"],
                   "step": "fa_create_block_mask + fa_flex_forward", "out": "fp32 O, fp32 LSE",
                   "l2": "inputs larger than the 129 MB L2 (no flush)",
                   "parallelism": "1 GPU" if world == 1 else
                   f"{world} ranks, batch x{world}, partitioned by (batch row, KV head) units, no collective"},
    }
    line.update({k_: v_ for k_, v_ in summ.items() if k_ != "workload"})
    line.update({
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps * step_launches,
        "clocks": clk.summary(), "status": fa.status_string(st_code), "wall_s": wall,
    })
    if others:
        line["prefill_workloads"] = others
    if split_line:
        line["split_prefill"] = split_line
    if dec_line:
        line["decode"] = dec_line
    if bwd_line:
        line["backward"] = bwd_line
    if paged_line:
        line["paged_prefill"] = paged_line
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def pf_config(w):
    return f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} N={w.q_len} d={w.d} Bq=Bk={w.bq}"


def bench_backward(args, dev, pk, w, q, k, v, bm, sc, out, lse, phys_flops):
    """fa_flex_backward (delta, dQ and dK/dV kernels) on the forward's own mask, O and LSE. Algorithmic
    FLOPs are 2.5x the forward's visited-block FLOPs (S recompute, dP, dV, dK, dQ: five d-deep products
    per visited pair against the forward's two)."""
    import torch

    from block_sparse_masked_create_gb300 import fa, workloads
    dout = workloads.bf16_torch(w.dout_bits(), dev)
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
    dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
    delta = torch.empty(lse.shape, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def bwd():
        fa.flex_backward(q, k, v, out, lse, dout, bm, sc, w.scale, dq=dq, dk=dk, dv=dv, delta=delta, status=status)

    for _ in range(3):
        bwd()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    n = max(3, args.steps // 2)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        bwd()
        b.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    med = statistics.median(ms)
    flop = 2.5 * phys_flops
    tf = flop / (med * 1e-3) / 1e12
    return {"workload": f"{w.name} backward: dout ~ N(0,1) bf16, dq/dk/dv fp32",
            "kernels": "delta + dQ (row lists) + dK/dV (query-side transpose); tcgen05 for 128x128 blocks",
            "ms_median": med, "algorithmic_tflop": flop / 1e12, "tflops": tf, "pct_bf16_peak": tf / pk["bf16"],
            "peak_src": f"{pk['src']} bf16 burst", "launches_per_step": 3,
            "status": fa.status_string(fa.check_status(status))}


def time_events(fn, n, stream):
    """Median milliseconds of fn() over n launches, CUDA events on `stream` after 3 warm-up calls."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def bench_split_prefill(args, dev, pk, q_len=256, kv_len=131072, H=8, chunk=64):
    """fa_flex_forward_split against fa_flex_forward on a chunked prefill: q_len new tokens at the end of a
    kv_len-token context (causal in global positions, query offset kv_len - q_len), B = 1, Hq = Hkv = H,
    d = 128, 128 x 128 blocks. Unsplit, each CTA walks two whole rows of ~kv_len / 128 key blocks and only
    H * ceil(q_len / 256) CTAs exist; split into chunks of `chunk` key blocks, the rows spread over the GPU."""
    import numpy as np
    import torch

    from block_sparse_masked_create_gb300 import fa, workloads
    w = workloads.Prefill("chunked_prefill", 1, H, H, q_len, kv_len, 128, 128, 128, [("causal",)], {},
                          1.0 / math.sqrt(128), 0x5EED0010).generate()
    q = workloads.bf16_torch(w.q_bits, dev)
    k = workloads.bf16_torch(w.k_bits, dev)
    v = workloads.bf16_torch(w.v_bits, dev)
    off = torch.tensor([kv_len - q_len], dtype=torch.int32, device=dev)
    rule = fa.make_mask_rule(w.rule, q_offset=off, batch_dependent=True)
    bm = fa.create_block_mask(rule, 1, H, q_len, kv_len, 128, 128, device=dev, keep=[off])
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((1, H, q_len), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.forward_split_workspace_bytes(bm, 1, H, 128, chunk), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    st = fa.block_mask_stats(bm).cpu().tolist()
    flop = 4.0 * 128 * 128 * 128 * (st[0] + st[1]) * H
    stream = torch.cuda.current_stream(dev)
    steps = max(5, args.steps)
    ms_plain = time_events(lambda: fa.flex_forward(q, k, v, bm, None, w.scale, out=out, lse=lse, status=status),
                           steps, stream)
    ms_split = time_events(lambda: fa.flex_forward_split(q, k, v, bm, None, w.scale, chunk_blocks=chunk, out=out,
                                                         lse=lse, workspace=ws, status=status), steps, stream)
    tf_split = flop / (ms_split * 1e-3) / 1e12
    return {"workload": f"chunked prefill: {q_len} new tokens after a {kv_len - q_len}-token context, B=1 "
                        f"Hq=Hkv={H} d=128, causal in global positions, 128x128 blocks; chunks of {chunk} key blocks",
            "rows_max_blocks": st[3], "forward_ms_median": ms_plain, "split_ms_median": ms_split,
            "forward_tflops": flop / (ms_plain * 1e-3) / 1e12, "split_tflops": tf_split,
            "split_pct_bf16_peak": tf_split / pk["bf16"], "speedup": ms_plain / ms_split,
            "launches_split": 3, "status": fa.status_string(fa.check_status(status))}


def bench_paged_prefill(args, dev, pk, w, q, bm, sc, phys_flops):
    """fa_flex_forward_paged on the workload's own mask: K and V split into 128-token pages stored at
    shuffled physical ids (one page per key block), against the contiguous forward timed the same way."""
    import torch

    from block_sparse_masked_create_gb300 import fa, workloads
    kpb, table = workloads.paged_kv(w.k_bits, 128, w.seed)
    vpb, _ = workloads.paged_kv(w.v_bits, 128, w.seed)
    kp = workloads.bf16_torch(kpb, dev)
    vp = workloads.bf16_torch(vpb, dev)
    pt = torch.from_numpy(table).to(dev)
    k = workloads.bf16_torch(w.k_bits, dev)
    v = workloads.bf16_torch(w.v_bits, dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.Hq, w.q_len), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    n = max(5, args.steps)
    ms_p = time_events(lambda: fa.flex_forward_paged(q, kp, vp, pt, bm, w.kv_len, sc, w.scale, out=out, lse=lse,
                                                     status=status), n, stream)
    ms_c = time_events(lambda: fa.flex_forward(q, k, v, bm, sc, w.scale, out=out, lse=lse, status=status), n, stream)
    tf = phys_flops / (ms_p * 1e-3) / 1e12
    return {"workload": f"{w.name} with K/V in 128-token pages at shuffled physical ids ({kpb.shape[0]} pages)",
            "ms_median": ms_p, "tflops": tf, "pct_bf16_peak": tf / pk["bf16"],
            "contiguous_ms_median": ms_c, "paged_over_contiguous": ms_p / ms_c,
            "status": fa.status_string(fa.check_status(status))}


def bench_decode(args, dev, pk):
    import numpy as np
    import torch

    from block_sparse_masked_create_gb300 import fa, workloads
    d = workloads.cfg5(Bz=args.decode_requests).generate()
    q = workloads.bf16_torch(d.q_bits, dev)
    kp = workloads.bf16_torch(d.k_bits, dev)
    vp = workloads.bf16_torch(d.v_bits, dev)
    pt = torch.from_numpy(d.page_table).to(dev)
    off = torch.from_numpy(d.q_offset).to(dev)
    rule = fa.make_mask_rule(d.rule, q_offset=off, batch_dependent=True)
    bm = fa.create_block_mask(rule, d.Bz, d.Hq, 1, d.kv_len, 1, d.page, device=dev, keep=[off])
    out = torch.empty_like(q)
    lse = torch.empty((d.Bz, d.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.decode_workspace_bytes(d.Bz, d.Hq, d.d, d.max_pages, d.page), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        fa.flex_decode(q, kp, vp, pt, bm, None, d.scale, out=out, lse=lse, workspace=ws, status=status)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    n = max(5, args.steps)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        fa.flex_decode(q, kp, vp, pt, bm, None, d.scale, out=out, lse=lse, workspace=ws, status=status)
        b.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    # per-step decode table: a fresh one-row build vs the row selection from a table prebuilt once for the
    # longest context (global positions, 128-row query blocks)
    L = d.kv_len
    big = fa.create_block_mask(fa.make_mask_rule(d.rule), 1, d.Hq, L, L, 128, d.page, device=dev)
    sel = fa.select_rows(big, off)
    ms_build = time_events(lambda: fa.recreate_block_mask(bm, rule, d.Bz, d.Hq, 1, d.kv_len, 1, d.page), n, stream)
    ms_sel = time_events(lambda: fa.select_rows(big, off, out=sel), n, stream)
    kv_bytes = int(sum(int(L) for L in d.kv_lens)) * d.Hkv * d.d * 2 * 2
    other = q.numel() * 2 + out.numel() * 2 + lse.numel() * 4 + pt.numel() * 4
    med = statistics.median(ms)
    gbs = (kv_bytes + other) / (med * 1e-3) / 1e9
    return {"workload": f"cfg5 paged decode: {d.Bz} requests, Hq=32, Hkv=8, d=128, 128-token pages, L~U[1024,32768]",
            "kv_gb": kv_bytes / 1e9, "ms_median": med, "GB/s": gbs, "pct_hbm": gbs / pk["hbm"],
            "step_mask_build_us": 1e3 * ms_build, "step_mask_from_prebuilt_us": 1e3 * ms_sel,
            "status": fa.status_string(fa.check_status(status)),
            "note": "KV read once per KV head; K/V pages 2x%.1f GB > L2" % (d.k_bits.nbytes / 1e9)}


def load_traffic(wl):
    """DRAM bytes per launch of the forward kernel from the committed ncu capture, or None when there is no
    capture for this workload or the kernel's sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        h = hashlib.sha1()
        for name in ("fwd_tc5.cu", "fa_internal.cuh"):
            with open(os.path.join(ROOT, "block_sparse_masked_create_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != t.get("source_sha1"):
            return None
        return t.get(wl)
    except Exception:
        return None


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if args.decode_only:
        import torch
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        print(json.dumps(bench_decode(args, dev, peaks())), flush=True)
        return
    ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()

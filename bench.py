"""Benchmark: absorbed MLA decode at V3 geometry (H=128, B=64, S=4096, T=1).

One step = one pass of the whole hot path through libmla.so: split plan,
absorption (q_nope @ W_UK), split-KV latent attention (with the LSE merge of
split groups in the same kernel), un-absorption (o_lat @ W_UV).  The step is captured into one
CUDA graph so that host launch cost does not pace the GPU; the dominant
kernel is timed separately: a decode-only graph (eight chained decode launches,
one when the L2 is flushed between launches) bracketed by CUDA events on the
launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload uniform|tiny|ragged|long|extend|sparse] [--T T] [--splits N]
                  [--arm absorb|normal]

The default workload is the uniform V3 batch; the others (the tiny V2-Lite
case, the ragged batch, the single 131072-row sequence with --splits N, the
causal extend batch with --T new rows) print the same JSON line for that
workload.  ``--arm normal`` times the decompressed comparison arm (expansion
of the latent cache into per-head keys and values, then causal MHA) on the
same workload instead.  ``--workload sparse`` times the index-driven decode
(mla_decode_sparse) on its own: 64 sequences of 8192 cached rows, one query
token each, top-2048 lists of distinct rows in random order.  A workload whose
cache fits in L2 is timed with an L2 flush between steps, outside the timed
events: a 256 MB write, then a 256 MB read, so that the L2 holds none of the
workload's lines and no dirty lines of the flush either (their write-back
would otherwise take HBM bandwidth inside the timed region: measured 53.9
against 49.2 us per launch on the long-context decode).

Multi-GPU runs are replicas: each rank runs the same independent batch (the
path shards by request and needs no collective); ``value`` is the tokens of
all ranks divided by the slowest rank's time.  ``--impl reference`` times the
float64 CPU oracle on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_INDEX = 2
WORKLOADS = {"tiny": 1, "uniform": 2, "ragged": 3, "long": 4, "extend": 5, "sparse": 6}
SPARSE = {"H": 128, "B": 64, "S_q": 1, "topk": 2048, "ctx": 8192, "seed": 1206}
METRIC = "MLA decode tokens/s and achieved HBM GB/s (% of roofline) at V3 geometry"
L2_BYTES = 129 * 2**20


class L2Flush:
    """Evicts the L2 between timed launches: a 256 MB write (the workload's lines
    leave the cache) followed by a 256 MB read (the flush's own dirty lines are
    written back before the timed region, not during it)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 * 2**20, dtype=torch.float32, device=dev)
        self.acc = torch.empty(1, dtype=torch.float32, device=dev)

    def __call__(self, i: int):
        import torch
        self.w.fill_(i & 0xff)
        torch.sum(self.r, dim=0, out=self.acc)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


PROFILE = os.path.join(ROOT, "profiles", "decode_sm103_v3_uniform_b64_s4096.md")
DECODE_SOURCES = ["mla_latent_cache_gb300/csrc/mla_decode_sm103.cu", "mla_latent_cache_gb300/csrc/sm103_ptx.cuh",
                  "mla_latent_cache_gb300/csrc/mla_internal.cuh", "mla_latent_cache_gb300/csrc/mla_plan_merge.cuh"]


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, or None when the
    decode kernel's sources changed since that capture."""
    import hashlib
    import re
    if not os.path.exists(PROFILE):
        return None
    text = open(PROFILE).read()
    m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch\s*\|\s*(\d+)", text)
    if not m_sha or not m_bytes:
        return None
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return int(m_bytes.group(1)) if h.hexdigest()[:16] == m_sha.group(1) else None


def algorithmic_bytes(w, row_bytes: int = 1152) -> dict:
    """Bytes each kernel of the step must move at minimum (inputs read once, outputs written once);
    row_bytes: one cached row (1152 bf16, 656 in the FP8 format)."""
    H, B, T = w.H, w.B, w.T
    rows = int(w.seq_lens.astype(np.int64).sum())
    BT = B * T
    decode = rows * row_bytes + BT * H * (512 + 64) * 2 + BT * H * 512 * 2 + BT * H * 4 + w.block_table.size * 4 + B * 4
    absorb = BT * H * 128 * 2 + H * 128 * 512 * 2 + BT * H * 512 * 2
    unabsorb = BT * H * 512 * 2 + H * 128 * 512 * 2 + BT * H * 128 * 2
    return {"decode": decode, "absorb": absorb, "unabsorb": unabsorb, "step": decode + absorb + unabsorb}


def algorithmic_flops(w) -> dict:
    H = w.H
    from_pairs = 0
    for S in w.seq_lens:
        S = int(S)
        for t in range(w.T):
            lim = S if not w.causal else max(0, min(S, S - w.T + t + 1))
            from_pairs += lim
    decode = 2 * H * from_pairs * (576 + 512)
    bmm = 2 * 2 * w.B * w.T * H * 128 * 512
    return {"decode": decode, "bmm": bmm, "step": decode + bmm}


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}_{id(self)}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.5)   # let it start sampling before the timed region begins
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, *others: "ClockSampler") -> dict:
        """Median SM clock, maximum clock and throttle reasons over this sampler's
        samples and those of `others` (further timed regions of the same run)."""
        sm, smax, reasons, ok = [], [], set(), False
        for smp in (self,) + others:
            if smp._collect(sm, smax, reasons):
                ok = True
        if not ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}

    def _collect(self, sm, smax, reasons) -> bool:
        if self.proc is None or not os.path.exists(self.path):
            return False
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return True


def cpu_oracle_sample(w, budget_s: float = 15.0):
    """Time the float64 oracle (absorb + latent attention + un-absorb) on whole sequences of the
    workload until ~budget_s of CPU work; returns (tokens/s, sequences done, seconds, cores)."""
    from mla_latent_cache_gb300 import workloads as W
    from oracle import mla_oracle as O
    pool, bt = w.compact_view()
    f = W.bf16_bits_to_f64
    q_nope, q_pe, w_uk, w_uv = f(w.q_nope), f(w.q_pe), f(w.w_uk), f(w.w_uv)
    done = 0
    t0 = time.perf_counter()
    while done < w.B:
        b = done
        n = (int(w.seq_lens[b]) + 63) // 64
        local_pool = f(pool[bt[b, :n]])          # this sequence's blocks, widened to float64
        local_bt = np.arange(n, dtype=np.int64)[None]
        O.absorbed_layer_ref(q_nope[[b]], q_pe[[b]], local_pool, local_bt, w.seq_lens[[b]], w_uk, w_uv, w.causal)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info
        threads = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        threads = cores
    return done * w.T / dt, done, dt, min(cores, threads) if threads else cores


def max_over_ranks(x: float, device=None) -> float:
    """The slowest rank's value (replicas are timed by the slowest one): an all-reduce
    MAX over the process group, the identity when there is none."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput of `world` replicas: every rank's units over the slowest time."""
    return units_per_rank * world / (ms / 1000.0)


def _emit(line: dict):
    print(json.dumps(line), flush=True)


def workload_config(w, args, world: int) -> dict:
    """The workload keys both arms print (the reference arm runs a bounded sample of it)."""
    fp8 = getattr(args, "cache", "bf16") == "fp8"
    pool_bytes = w.num_blocks * 64 * (656 if fp8 else 1152)
    extra = {"cache": "fp8 656-byte rows (E4M3 latent, 4 fp32 scales, bf16 RoPE)"} if fp8 else {}
    return {**extra, "workload": w.name, "H": w.H, "B": w.B, "T": w.T, "S": int(w.seq_lens[0]),
            "S_total": int(np.asarray(w.seq_lens, dtype=np.int64).sum()), "page": 64, "pool_blocks": w.num_blocks,
            "parallelism": f"replicas{world}", "splits": args.splits or "auto",
            "l2": ("L2 flushed between steps (256 MB write then 256 MB read, outside the timed events)" if pool_bytes < 2 * L2_BYTES
                   else f"inputs larger than L2: {pool_bytes / 1e6:.0f} MB latent pool vs 129 MB L2")}



def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    from mla_latent_cache_gb300 import workloads as W
    w = W.config_workload(WORKLOADS[args.workload], T=args.T if args.workload == "extend" else None)
    per_step = []
    samples = []
    for _ in range(args.warmup):
        cpu_oracle_sample(_one_seq(w), budget_s=0.0)
    budget = min(args.ref_budget, 120.0 / max(1, args.steps))   # whole run stays within a few minutes
    for _ in range(args.steps):
        tps, done, dt, cores = cpu_oracle_sample(w, budget_s=budget)
        per_step.append(dt)
        samples.append((tps, done, dt, cores))
    tps = sum(s[1] for s in samples) * w.T / sum(per_step)
    cores = samples[-1][3]
    seqs = [s[1] for s in samples]
    # ms_per_step is the time each timed step actually took: one bounded sample of
    # the workload (its first sequences, whole), not the full batch
    ms = 1000.0 * sum(per_step) / len(per_step)
    _emit({"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(w, args, world),
           "step": f"one bounded sample of the workload per step: its first sequences, whole "
                   f"({min(seqs)}-{max(seqs)} of B={w.B}), absorb + attention + un-absorb in float64",
           "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": f"{min(seqs)}-{max(seqs)} whole sequences of the workload per step "
                                      f"(~{budget:.1f} s budget per step)"},
           "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})
    return 0


def _one_seq(w):
    from mla_latent_cache_gb300 import workloads as W
    return W.custom_workload(w.H, [64], T=1, seed=1)


def run_ours(args):
    import torch
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from mla_latent_cache_gb300 import binding as L
    from mla_latent_cache_gb300 import workloads as W
    from mla_latent_cache_gb300.runtime import DecodeStep

    w = W.config_workload(WORKLOADS[args.workload], T=args.T if args.workload == "extend" else None)
    st = DecodeStep(w, device=dev, num_splits_override=args.splits, cache_format=args.cache)
    stream = torch.cuda.Stream(device=dev)
    row_bytes = 656 if args.cache == "fp8" else 1152
    pool_bytes = w.num_blocks * 64 * row_bytes
    flush = L2Flush(dev) if pool_bytes < 2 * L2_BYTES else None
    hbm_peak, tc_peak, peak_kind = _peaks()
    ab = algorithmic_bytes(w, row_bytes)
    fl = algorithmic_flops(w)

    # warm up eagerly once (sets kernel attributes), then capture
    with torch.cuda.stream(stream):
        st.step(stream)
    stream.synchronize()
    # One graph per step: plan, absorb, decode (+ merge), un-absorb on one stream,
    # every kernel chained to its predecessor with programmatic dependent launch
    # (the absorption streams its weights in while the plan runs).  A second graph
    # holds decode launches alone, replayed between CUDA events to time the dominant kernel.
    g_step, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        st.step(stream)
    # Decode launches per decode graph: eight back to back (chained by
    # programmatic launch, as a model chains its layers' decodes), so that the
    # graph's own launch latency is not charged to the kernel (measured: 67.6 us
    # per launch with four, 67.1-67.3 with eight or sixteen); one when the pool is
    # small enough that the L2 has to be flushed between launches.
    dec_per_graph = 1 if flush is not None else 8
    with torch.cuda.graph(g_dec, stream=stream):
        for _ in range(dec_per_graph):
            st.decode(stream)
    launches_per_step = 4  # plan, absorb, decode (its merge runs in the same kernel), un-absorb

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g_step.replay()
            g_dec.replay()
    stream.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    step_evs = [(ev(), ev()) for _ in range(args.steps)] if flush is not None else None
    t_start, t_end = ev(), ev()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # The decode alone first, for the kernel roofline (same inputs, same launch
        # configuration), before the long step loop: it is compared with the copy
        # peak measured as a burst, so it is timed as a kernel alone, not after
        # minutes of power-capped load.
        dec_steps = max(1, args.dec_steps)   # replays of the decode-only graph (whatever --steps is: a stable kernel figure)
        evs = [(ev(), ev()) for _ in range(dec_steps)]
        with torch.cuda.stream(stream):
            for i in range(dec_steps):
                if flush is not None:
                    flush(i)
                evs[i][0].record(stream)
                g_dec.replay()
                evs[i][1].record(stream)
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(args.steps):
                if flush is not None:
                    flush(i)                       # evict the cache lines of the previous step
                    step_evs[i][0].record(stream)
                g_step.replay()
                if flush is not None:
                    step_evs[i][1].record(stream)
            t_end.record(stream)
        stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    dec_ms = sum(a.elapsed_time(b) for a, b in evs) / dec_steps / dec_per_graph
    if flush is not None:
        ms = sum(a.elapsed_time(b) for a, b in step_evs) / args.steps
    else:
        ms = total_ms / args.steps
    ms = max_over_ranks(ms, dev)
    value = replica_throughput(w.B * w.T, world, ms)
    status, info = L.mla_read_device_status(st.workspace, stream)
    if status != L.MLA_OK:
        raise RuntimeError(f"device status after timing: {L.mla_status_string(status)} ({info})")

    # end to end through the C ABI with host buffers: every step copies its inputs
    # (q_nope, q_pe, seq_lens, block table: one pinned host buffer mirroring the
    # device buffer they live in) to the device and reads its o back.  Two input
    # buffers and two outputs alternate, so that the upload of the next step and
    # the read-back of the previous one run on side streams under the current
    # step's kernels; one graph holds two steps (buffer sets A and B).
    io_a = st.io_set()
    io_b = st.new_io_set()
    h_in = torch.empty_like(st.inputs, device="cpu").pin_memory(); h_in.copy_(st.inputs)
    h_o = [torch.empty_like(st.o, device="cpu").pin_memory() for _ in range(2)]
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_o[0].numel() * h_o[0].element_size()
    e_pairs = max(2, min(args.steps, 200) // 2)
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    g_e2e = torch.cuda.CUDAGraph()

    def half(io_run, io_next, h_out_prev, o_prev):
        fork = torch.cuda.Event()
        fork.record(stream)
        up, down = torch.cuda.Event(), torch.cuda.Event()
        s_up.wait_event(fork)
        with torch.cuda.stream(s_up):
            io_next["inputs"].copy_(h_in, non_blocking=True)      # the next step's inputs
            up.record(s_up)
        s_down.wait_event(fork)
        with torch.cuda.stream(s_down):
            h_out_prev.copy_(o_prev, non_blocking=True)           # the previous step's output
            down.record(s_down)
        st.bind(io_run)
        st.step(stream)
        stream.wait_event(up)
        stream.wait_event(down)

    with torch.cuda.graph(g_e2e, stream=stream):
        half(io_a, io_b, h_o[1], io_b["o"])
        half(io_b, io_a, h_o[0], io_a["o"])
    st.bind(io_a)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_e2e.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local) as clocks_e2e:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(e_pairs):
                g_e2e.replay()
            e1.record(stream)
        stream.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / (2 * e_pairs), dev)
    e2e_value = replica_throughput(w.B * w.T, world, e2e_ms)
    # (each step's output lands on the host one step later: o of the last step of
    # a replay is read back in the next replay's first half)
    e2e_check = bool(torch.equal(h_o[0].to(dev), io_a["o"]) and torch.equal(h_o[1].to(dev), io_b["o"]))

    achieved = ab["decode"] / (dec_ms / 1000.0) / 1e9
    tflops = fl["decode"] / (dec_ms / 1000.0) / 1e12
    ridge = tc_peak * 1e12 / (hbm_peak * 1e9)
    if fl["decode"] / ab["decode"] > ridge:
        roof = {"bound": "tensor", "kernel": "mla_decode (split-KV decode + merge)", "achieved": tflops,
                "peak": tc_peak, "peak_kind": peak_kind, "unit": "TFLOP/s", "frac": tflops / tc_peak,
                "traffic": None, "algorithmic_flops": fl["decode"], "decode_ms": dec_ms, "decode_gbs": achieved}
    else:
        roof = {"bound": "hbm", "kernel": "mla_decode (split-KV decode + merge)", "achieved": achieved,
                "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm_peak,
                "traffic": (profiled_traffic() if WORKLOADS[args.workload] == WORKLOAD_INDEX and args.cache == "bf16"
                            else None),
                "algorithmic_bytes": ab["decode"], "decode_ms": dec_ms, "decode_tflops": tflops}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, args, world),
        "step": "plan, absorb, decode (the split plan's merge in the same kernel), unabsorb; one CUDA graph per "
                "step, kernels chained with programmatic dependent launch; the decode timed alone in its own "
                f"graph ({dec_per_graph} chained launches per replay, {dec_steps} replays, before the step loop)",
        "roofline": roof,
        "step_hbm_gbs": ab["step"] / (ms / 1000.0) / 1e9,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "overlap": "uploads and read-backs on side streams under the other "
                                                  "buffer set's step (two input buffers, two outputs)",
                "readback_matches_device": e2e_check},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(clocks_e2e),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, done, dt, cores = cpu_oracle_sample(w, budget_s=args.ref_budget)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{done} whole sequences of the workload (absorb + attention + "
                                          f"un-absorb, float64) in {dt:.1f} s"}
    if rank == 0:
        _emit(line)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def normal_flops_bytes(w) -> dict:
    """Algorithmic FLOPs and bytes of the Normal arm's two kernels."""
    H, rows = w.H, int(np.asarray(w.seq_lens, dtype=np.int64).sum())
    pairs = 0
    for S in w.seq_lens:
        S = int(S)
        for t in range(w.T):
            pairs += S if not w.causal else max(0, min(S, S - w.T + t + 1))
    BT = w.B * w.T
    expand_f = 2 * rows * 512 * 256 * H
    attn_f = 2 * H * pairs * (192 + 128)
    expand_b = rows * 512 * 2 + 2 * H * 128 * 512 * 2 + rows * H * 256 * 2
    attn_b = rows * H * 256 * 2 + rows * 64 * 2 + BT * H * (128 + 64 + 128) * 2 + BT * H * 4
    return {"expand_flops": expand_f, "attn_flops": attn_f, "expand_bytes": expand_b, "attn_bytes": attn_b}


def run_normal(args):
    """The Normal (decompressed) arm on the same workload: expansion + causal MHA."""
    import torch
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from mla_latent_cache_gb300 import binding as L
    from mla_latent_cache_gb300 import workloads as W
    from mla_latent_cache_gb300.runtime import NormalStep
    w = W.config_workload(WORKLOADS[args.workload], T=args.T if args.workload == "extend" else None)
    st = NormalStep(w, device=dev, chunk_rows=args.chunk)
    stream = torch.cuda.Stream(device=dev)
    hbm_peak, tc_peak, peak_kind = _peaks()
    nf = normal_flops_bytes(w)
    with torch.cuda.stream(stream):
        st.step(stream)
    stream.synchronize()
    if args.chunk > 0:
        return _run_normal_chunked(args, w, st, stream, nf, tc_peak, peak_kind, local)
    g_exp, g_att = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_exp, stream=stream):
        st.expand(stream)
    with torch.cuda.graph(g_att, stream=stream):
        st.attention(stream)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g_exp.replay(); g_att.replay()
    stream.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    marks = [(ev(), ev(), ev()) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                marks[i][0].record(stream)
                g_exp.replay()
                marks[i][1].record(stream)
                g_att.replay()
                marks[i][2].record(stream)
        stream.synchronize()
    exp_ms = sum(a.elapsed_time(b) for a, b, _ in marks) / args.steps
    att_ms = sum(b.elapsed_time(c) for _, b, c in marks) / args.steps
    ms = exp_ms + att_ms
    status, info = L.mla_read_device_status(None, stream)
    if status != L.MLA_OK:
        raise RuntimeError(f"device status after timing: {L.mla_status_string(status)} ({info})")
    tokens = w.B * w.T
    exp_tf = nf["expand_flops"] / (exp_ms / 1e3) / 1e12
    att_tf = nf["attn_flops"] / (att_ms / 1e3) / 1e12
    dominant = ("mla_normal_expand", exp_tf, exp_ms) if exp_ms >= att_ms else ("mla_normal_attention", att_tf, att_ms)
    line = {
        "impl": "ours", "arm": "normal", "metric": METRIC, "value": tokens / (ms / 1e3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "H": w.H, "B": w.B, "T": w.T, "S": int(w.seq_lens[0]), "page": 64,
                   "step": "expand (latent -> per-head k_nope, v) + causal MHA, CUDA graphs",
                   "l2": "inputs larger than L2 (expanded keys/values: %.0f MB)" % (st.kv_exp.numel() * 2 / 1e6)},
        "roofline": {"bound": "tensor", "kernel": dominant[0], "achieved": dominant[1], "peak": tc_peak,
                     "peak_kind": peak_kind, "unit": "TFLOP/s", "frac": dominant[1] / tc_peak, "traffic": None},
        "kernels": {"expand_ms": exp_ms, "expand_tflops": exp_tf,
                    "expand_gbs": nf["expand_bytes"] / (exp_ms / 1e3) / 1e9,
                    "attention_ms": att_ms, "attention_tflops": att_tf,
                    "attention_gbs": nf["attn_bytes"] / (att_ms / 1e3) / 1e9},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
    }
    _emit(line)
    return 0


def sparse_bytes(sw) -> int:
    """Algorithmic bytes of one sparse decode: the listed rows (1152 B each, read once per
    token that lists them), the lists, the query and the outputs."""
    n = int(sum(min(int(sw.topk_length[b]), sw.topk) for b in range(sw.B))) * sw.S_q
    BT = sw.B * sw.S_q
    return n * 1152 + n * 4 + BT * sw.H * (576 * 2 + 512 * 2 + 4) + sw.B * 4


def run_sparse(args):
    """The index-driven decode alone: device-resident inputs (L2 flushed between launches),
    and end to end with the step's query, lists and lengths copied in and o_lat, lse read back."""
    import torch
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from mla_latent_cache_gb300 import binding as L
    from mla_latent_cache_gb300 import workloads as W
    from mla_latent_cache_gb300.runtime import SparseStep
    c = SPARSE
    sw = W.sparse_workload(c["H"], [c["ctx"]] * c["B"], c["S_q"], c["topk"], seed=c["seed"],
                           name=f"v32_sparse_b{c['B']}_sq{c['S_q']}_topk{c['topk']}_ctx{c['ctx']}")
    st = SparseStep(sw, device=dev, num_splits_override=args.splits)
    stream = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)
    hbm_peak, tc_peak, peak_kind = _peaks()
    nbytes = sparse_bytes(sw)
    with torch.cuda.stream(stream):
        st.decode(stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        st.decode(stream)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g.replay()
    stream.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    evs = [(ev(), ev()) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush(i)                           # the listed rows of the previous launch leave the L2
                evs[i][0].record(stream)
                g.replay()
                evs[i][1].record(stream)
        stream.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    status, info = L.mla_read_device_status(st.workspace, stream)
    if status != L.MLA_OK:
        raise RuntimeError(f"device status after timing: {L.mla_status_string(status)} ({info})")
    # end to end: pinned host copies of q_lat, q_pe, indices, lengths in; o_lat, lse out
    ins = [st.q_lat, st.q_pe, st.indices, st.topk_length]
    h_in = [torch.empty_like(t, device="cpu").pin_memory() for t in ins]
    for h, t in zip(h_in, ins):
        h.copy_(t)
    outs = [st.o_lat, st.lse]
    h_out = [torch.empty_like(t, device="cpu").pin_memory() for t in outs]
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        for t, h in zip(ins, h_in):
            t.copy_(h, non_blocking=True)
        st.decode(stream)
        for h, t in zip(h_out, outs):
            h.copy_(t, non_blocking=True)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_e2e.replay()
    stream.synchronize()
    e_steps = max(3, min(args.steps, 200))
    e0, e1 = ev(), ev()
    with ClockSampler(local) as clocks_e2e:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(e_steps):
                g_e2e.replay()
            e1.record(stream)
        stream.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    tokens = sw.B * sw.S_q
    achieved = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": tokens / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": sw.name, "H": sw.H, "B": sw.B, "S_q": sw.S_q, "topk": sw.topk, "ctx": c["ctx"],
                   "page": 64, "pool_blocks": sw.ctx.num_blocks, "parallelism": "replicas1",
                   "splits": args.splits or "auto",
                   "l2": "L2 flushed between launches (256 MB write then 256 MB read, outside the timed events)"},
        "step": "mla_decode_sparse (plan + index-driven decode with the in-kernel merge), one CUDA graph",
        "roofline": {"bound": "hbm", "kernel": "mla_decode_sparse", "achieved": achieved, "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": None,
                     "algorithmic_bytes": nbytes, "decode_ms": ms},
        "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in h_in),
                "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in h_out), "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(clocks_e2e),
    }
    _emit(line)
    return 0


def _run_normal_chunked(args, w, st, stream, nf, tc_peak, peak_kind, local):
    """The chunked-prefix Normal path: all windows (expand + attention each) in one graph."""
    import torch
    from mla_latent_cache_gb300 import binding as L
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        st.step(stream)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g.replay()
    stream.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                evs[i][0].record(stream)
                g.replay()
                evs[i][1].record(stream)
        stream.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    status, info = L.mla_read_device_status(None, stream)
    if status != L.MLA_OK:
        raise RuntimeError(f"device status after timing: {L.mla_status_string(status)} ({info})")
    flops = nf["expand_flops"] + nf["attn_flops"]
    tf = flops / (ms / 1e3) / 1e12
    windows = -(-w.max_pages * 64 // args.chunk)
    line = {
        "impl": "ours", "arm": "normal_chunked", "metric": METRIC, "value": w.B * w.T / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "H": w.H, "B": w.B, "T": w.T, "S": int(w.seq_lens[0]), "page": 64,
                   "chunk_rows": args.chunk, "windows": windows,
                   "step": "per window: expand its latents, attend to its keys, LSE-merge into the running "
                           "state; all windows in one CUDA graph",
                   "l2": "expanded window %.0f MB (whole prefix one-shot: %.0f MB)" % (
                       st.kv_exp.numel() * 2 / 1e6, w.H * w.B * (-(-w.max_pages // 2) * 128) * 512 / 1e6)},
        "roofline": {"bound": "tensor", "kernel": "mla_normal_chunked (expand + attention, all windows)",
                     "achieved": tf, "peak": tc_peak, "peak_kind": peak_kind, "unit": "TFLOP/s",
                     "frac": tf / tc_peak, "traffic": None},
        "gpu_launches": 2 * windows * args.steps,
        "clocks": clocks.summary(),
    }
    _emit(line)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-budget", type=float, default=15.0, help="seconds of CPU oracle work per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dec-steps", type=int, default=200,
                    help="replays of the decode-only graph timed for the roofline (a small count keeps a profiler's launch list on the step)")
    ap.add_argument("--workload", choices=sorted(WORKLOADS, key=WORKLOADS.get), default="uniform")
    ap.add_argument("--T", type=int, default=1, help="new rows per sequence (extend workload)")
    ap.add_argument("--splits", type=int, default=0, help="split count override (0 = the automatic plan)")
    ap.add_argument("--cache", choices=["bf16", "fp8"], default="bf16",
                    help="cache row format of the absorbed decode (fp8: 656-byte rows, mla_decode_fp8)")
    ap.add_argument("--chunk", type=int, default=0,
                    help="normal arm: chunked-prefix windows of this many cache rows (multiple of 128; 0 = one shot)")
    ap.add_argument("--arm", choices=["absorb", "normal"], default="absorb",
                    help="absorb: the latent-cache path (default); normal: the decompressed comparison arm")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "sparse":
        return run_sparse(args)
    if args.arm == "normal":
        return run_normal(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

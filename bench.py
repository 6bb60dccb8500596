"""KDA benchmark: prefill head-tokens/s (H*T per second) and decode GB/s at
D=128, each against the GB300 roofline.

A step is one chunked prefill of the mid-size workload (B=1, H=32,
T=8192, D=128, bf16 q/k/v/beta, fp32 g and state, chunk 64) with its inputs
resident in HBM (they total ~400 MB, larger than the 129 MB L2, so no L2
flush is needed between steps). The decode workload (B=256 sequences x 96
heads, 64 single-token steps on a 1.6 GB fp32 state, replayed from a CUDA
graph) is measured alongside and reported under "decode".

Prints ONE JSON line (rank 0). With --impl reference it times the fp64 CPU
oracle instead, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D = 128
C = 64
PREFILL = dict(H=32, T=8192, seed=1001)
DECODE = dict(B=256, H=96, steps=64, seed=1002)
WORKLOAD = "prefill_mid_bf16: B=1, H=32, T=8192, D=128, chunk=64, bf16 q/k/v/beta, fp32 g/state"
METRIC = "KDA prefill Mtok/s (H*T per s) at D=128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def prefill_bytes_per_head_token(io_bytes=2):
    """Minimal fused HBM traffic per head-token: q, k, v, out in the I/O type,
    g in fp32, beta in the I/O type."""
    return 4 * D * io_bytes + 4 * D + io_bytes


def prefill_flops_per_chunk(c=C, d=D):
    """12 C^3 + 8 C^2 D + 6 C D^2 per chunk and head ("Kimi K3: The Manos, The
    Mythos, The Legendos", section 复杂度分析)."""
    return 12 * c ** 3 + 8 * c * c * d + 6 * c * d * d


def decode_bytes_per_head_call(tokens=1, d=D):
    """Minimal HBM bytes per head and decode call of `tokens` tokens: the fp32
    state read and written once (~8 D^2, same section), plus each token's row
    (q, k, v, out in bf16, g in fp32, beta in bf16)."""
    return 8 * d * d + tokens * prefill_bytes_per_head_token()


def decode_flops_per_head_token(d=D):
    return 7 * d * d


def measured_traffic(key):
    """DRAM bytes per launch from a committed ncu capture, while the kernel
    source it was taken from is unchanged (else None)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            entry = json.load(f)[key]
        with open(os.path.join(ROOT, entry["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != entry["source_sha256_16"]:
                return None
        return entry
    except Exception:
        return None


def decode_traffic(units):
    """Decode DRAM bytes per launch, scaled by state count from the committed
    capture (traffic grows in proportion to the number of head states)."""
    e = measured_traffic("decode_b64_h96")
    if e is None:
        return None
    return e["bytes_per_launch"] * units / e["units_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                for k2, v in d.items():
                    if k2 == key or k2.startswith(key):
                        if isinstance(v, (int, float)):
                            out[key] = float(v)
                            break
            if "hbm_gbs" in out:
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def rank_seed(base, rank):
    """Each rank draws its own independent batch: the units shard across ranks
    with no exchange between them (weak scaling)."""
    return base + 7919 * rank


def max_over_ranks(x, world, device):
    """The largest value of x over all ranks (x itself on one rank): a step
    counts as done when the slowest rank is done."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, world, rank):
    """The oracle as it stands on the host cores, on bounded samples."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from kimi_delta_attention_rule_gb300 import inputs
    oracle.build()
    heads, toks = PREFILL["H"], 1024
    x = inputs.prefill_inputs([PREFILL["T"]], H=PREFILL["H"], io="bf16", seed=PREFILL["seed"])
    f = lambda t: t[:toks].float().numpy()
    q, k, v, g, b = f(x.q), f(x.k), f(x.v), f(x.g), x.beta[:toks].float().numpy()
    cores = oracle.default_threads()
    for _ in range(args.warmup):
        oracle.prefill(q, k, v, g, b, x.scale)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.prefill(q, k, v, g, b, x.scale)
        times.append(time.perf_counter() - t0)
    units = heads * toks
    sec = sum(times) / len(times)
    val = units / sec / 1e6
    sample = "first %d tokens x %d heads of the workload per step (fp64 oracle)" % (toks, heads)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "Mtok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": val, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "Mtok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def cpu_baseline(budget_s=10.0, max_reps=20):
    """Time the oracle as it stands on the prefill workload (all 32 heads x
    8192 tokens), repeated until about `budget_s` seconds of CPU time."""
    import oracle
    from kimi_delta_attention_rule_gb300 import inputs
    oracle.build()
    x = inputs.prefill_inputs([PREFILL["T"]], H=PREFILL["H"], io="bf16", seed=PREFILL["seed"])
    f = lambda t: t.float().numpy()
    args = (f(x.q), f(x.k), f(x.v), f(x.g), f(x.beta), x.scale)
    cores = oracle.default_threads()
    reps, total = 0, 0.0
    while total < budget_s and reps < max_reps:
        t0 = time.perf_counter()
        oracle.prefill(*args)
        total += time.perf_counter() - t0
        reps += 1
    units = reps * PREFILL["T"] * PREFILL["H"]
    return {"value": units / total / 1e6, "unit": "Mtok/s", "cores": cores, "kind": "oracle",
            "sample": "the full prefill workload (8192 tokens x 32 heads) %d times, %.1f s"
                      % (reps, total)}


def time_prefill_calls(call, stream, min_s=0.5, warm=2):
    """ms per call of `call()` on `stream` (CUDA events), over a number of calls
    fixed from one timed warm-up call so that the timed region lasts about min_s."""
    import torch
    for _ in range(warm):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    call()
    e1.record(stream)
    torch.cuda.synchronize()
    n = max(3, math.ceil(min_s * 1e3 / e0.elapsed_time(e1)))
    e0.record(stream)
    for _ in range(n):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n, n


def oracle_sample_rate(x, seqs, heads, max_tokens, init=None):
    """fp64 oracle head-tokens/s on a slice of a workload (host cores)."""
    import numpy as np
    import oracle
    oracle.build()
    cu = [0] + list(np.cumsum(x.lens))
    parts = [(cu[n], min(cu[n + 1], cu[n] + max_tokens)) for n in seqs]
    f = lambda t: np.concatenate([t[a:b][:, heads].float().cpu().numpy() for a, b in parts])
    lens = [b - a for a, b in parts]
    cus = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ini = None if init is None else init[seqs][:, heads].double().cpu().numpy()
    args = (f(x.q), f(x.k), f(x.v), f(x.g), f(x.beta), x.scale)
    t0 = time.perf_counter()
    oracle.prefill(*args, init_state=ini, cu_seqlens=cus)
    sec = time.perf_counter() - t0
    units = sum(lens) * len(heads)
    return {"value": units / sec / 1e6, "unit": "Mtok/s", "cores": oracle.default_threads(),
            "kind": "oracle", "sample": "%d tokens x %d heads of %d sequence(s), %.2f s"
            % (max(lens), len(heads), len(seqs), sec)}


def lpt_tail(chunks, nsm, longest_first=True):
    """Modelled share of the recurrence kernel's time in which some SMs are idle:
    chains of the given chunk counts started in order (longest first, or as
    given) on nsm SMs, one chain per SM at a time: 1 - total / (nsm * makespan)."""
    import heapq
    load = [0] * nsm
    heapq.heapify(load)
    for c in (sorted(chunks, reverse=True) if longest_first else chunks):
        heapq.heappush(load, heapq.heappop(load) + c)
    span = max(load)
    return 1.0 - sum(chunks) / (nsm * span) if span else 0.0


def bench_workloads(args, world, rank, dev, stream, peaks, peak_src):
    """The append-prefill (H=96) and packed varlen (64 sequences) workloads:
    Mtok/s, HBM roofline on minimal bytes, the pages' FLOP count against the
    bf16 peak, the schedule, and a sampled oracle rate."""
    import torch
    import kimi_delta_attention_rule_gb300 as kda
    from kimi_delta_attention_rule_gb300 import inputs
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    res = {}

    def bounded(run, ws_full, N, T, H, varlen, units, ms_full):
        """The same call with the ring-sized workspace (the fused schedule with
        per-chain rings of prepared blocks): its plan, time and throughput."""
        nb = kda.kda_prefill_workspace_size_ring(N, T, H, D, C, kda.KDA_BF16, varlen)
        if nb == 0 or nb >= ws_full.numel():
            return {"workspace_bytes": nb, "plan": "full workspace (no smaller plan)"}
        ws_r = torch.empty(nb, dtype=torch.uint8, device=dev)
        pl = kda.kda_prefill_plan(N, T, H, D, C, kda.KDA_BF16, varlen, nb)
        ms_r, n_r = time_prefill_calls(lambda: run(ws_r), stream)
        ms_r = max_over_ranks(ms_r, world, dev)
        assert kda.kda_workspace_status(ws_r) == kda.KDA_OK
        del ws_r
        return {"workspace_bytes": nb, "ms_per_call": ms_r, "calls_timed": n_r,
                "value": units / (ms_r * 1e-3) / 1e6, "unit": "Mtok/s",
                "vs_full_workspace": ms_full / ms_r,
                "plan": {"schedule": "fused", "groups": pl.groups,
                         "group_chains": pl.group_chains, "ring": pl.ring},
                "gpu_launches": n_r * (pl.groups + (1 if varlen else 0))}

    def line(name, desc, T_total, H, N, ms, calls, sched, extra):
        units = T_total * H * world
        state_bytes = 2 * N * H * D * D * 4  # initial state read, final state written
        byts = prefill_bytes_per_head_token() * T_total * H + state_bytes
        chunks = extra.pop("chunk_heads")
        gbs = byts / (ms * 1e-3) / 1e9
        tf = prefill_flops_per_chunk() * chunks / (ms * 1e-3) / 1e12
        res[name] = dict(workload=desc, value=units / (ms * 1e-3) / 1e6, unit="Mtok/s",
                         ms_per_call=ms, calls_timed=calls,
                         schedule={0: "split", 1: "fused"}[sched],
                         roofline={"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                                   "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                                   "peak_source": peak_src, "algorithmic_bytes_per_launch": byts},
                         tensor={"tflops_pages_count": tf, "peak": peaks["bf16_tflops"],
                                 "frac": tf / peaks["bf16_tflops"]},
                         gpu_launches=calls * (1 if sched == 1 else 2) + (calls if N > 1 else 0),
                         **extra)

    # append: a 32768-token prefill (untimed) gives the state; the 65536 new
    # tokens are the timed call
    w = inputs.WORKLOADS["append_h96"]
    P, Ta, Ha = w["prior"], w["T"], w["H"]
    x = inputs.prefill_inputs([P + Ta], H=Ha, io="bf16", seed=rank_seed(w["seed"], rank), device=dev)
    _, s_prior = kda.kda_prefill(x.q[:P], x.k[:P], x.v[:P], x.g[:P], x.beta[:P], x.scale, chunk=C)
    qa, ka, va, ga, ba = (t[P:] for t in (x.q, x.k, x.v, x.g, x.beta))
    out = torch.empty_like(qa)
    fin = torch.empty_like(s_prior)
    ws = kda.prefill_workspace(qa, None, N=1, T=Ta)
    sched = kda.kda_prefill_schedule(1, Ta, Ha, D, C, kda.KDA_BF16)
    run = lambda w_: kda.kda_prefill(qa, ka, va, ga, ba, x.scale, init_state=s_prior, chunk=C,
                                      out=out, final_state=fin, workspace=w_, stream=stream)
    ms, n = time_prefill_calls(lambda: run(ws), stream)
    ms = max_over_ranks(ms, world, dev)
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    extra = {"chunk_heads": Ha * (Ta // C), "workspace_bytes": ws.numel(),
             "bounded_workspace": bounded(run, ws, 1, Ta, Ha, False, Ta * Ha * world, ms)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        xs = inputs.PrefillInputs(qa, ka, va, ga, ba, None, None, x.scale, [Ta])
        extra["cpu_oracle"] = oracle_sample_rate(xs, [0], list(range(16)), 4096)
    line("append", "append_h96: H=96, D=128, fp32 state of a 32768-token prefill, then 65536 "
         "new bf16 tokens, chunk 64", Ta, Ha, 1, ms, n, sched, extra)
    del x, s_prior, qa, ka, va, ga, ba, out, fin, ws
    torch.cuda.empty_cache()

    # varlen: 64 packed sequences, lengths U[1024, 32768], H=32, g near the floor
    w = inputs.WORKLOADS["varlen64_h32_floor"]
    lens = inputs.varlen_lengths(w["n_seqs"], w["lo"], w["hi"], seed=w["seed"])
    x = inputs.prefill_inputs(lens, H=w["H"], io="bf16", seed=rank_seed(w["seed"], rank),
                              g_mode="floor", init="normal", device=dev)
    Nv, Hv, Tv = len(lens), w["H"], sum(lens)
    out = torch.empty_like(x.q)
    fin = torch.empty_like(x.init_state)
    ws = kda.prefill_workspace(x.q, x.cu_seqlens)
    sched = kda.kda_prefill_schedule(Nv, Tv, Hv, D, C, kda.KDA_BF16, True)
    run = lambda w_: kda.kda_prefill(x.q, x.k, x.v, x.g, x.beta, x.scale, init_state=x.init_state,
                                      cu_seqlens=x.cu_seqlens, chunk=C, out=out, final_state=fin,
                                      workspace=w_, stream=stream)
    ms, n = time_prefill_calls(lambda: run(ws), stream)
    ms = max_over_ranks(ms, world, dev)
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    chunks = [math.ceil(L / C) for L in lens]
    extra = {"chunk_heads": sum(chunks) * Hv, "workspace_bytes": ws.numel(),
             "bounded_workspace": bounded(run, ws, Nv, Tv, Hv, True, Tv * Hv * world, ms),
             "chains": Nv * Hv, "recurrence_tail_share_model": lpt_tail(chunks * Hv, nsm),
             "recurrence_tail_share_model_in_index_order":
                 lpt_tail([c for c in chunks for _ in range(Hv)], nsm, longest_first=False),
             "recurrence_order": "longest first (chunk-count classes)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        extra["cpu_oracle"] = oracle_sample_rate(x, [0], list(range(16)), 4096, init=x.init_state)
    line("varlen", "varlen64_h32_floor: 64 packed sequences, lengths U[1024, 32768] (%d tokens), "
         "H=32, D=128, bf16, g near the -5 floor, random initial states" % Tv, Tv, Hv, Nv, ms, n,
         sched, extra)
    del x, out, fin, ws
    torch.cuda.empty_cache()
    return res


def ncu_case(args):
    """A single kernel launched warmup + 1 times: the target of ncu captures."""
    import torch
    import kimi_delta_attention_rule_gb300 as kda
    from kimi_delta_attention_rule_gb300 import build as kbuild, inputs
    kbuild.build()
    kda.load()
    dev = torch.device("cuda", 0)
    if args.ncu_case == "layer":
        gen = torch.Generator(device=dev)
        gen.manual_seed(PREFILL["seed"] + 11)
        T, H = PREFILL["T"], PREFILL["H"]
        raw = [torch.randn((T, H, D), generator=gen, device=dev).to(torch.bfloat16)
               for _ in range(5)]
        braw = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
        convs = [0.5 * torch.randn((H, D, 4), generator=gen, device=dev) for _ in range(3)]
        nw = torch.ones(D, device=dev)
        for _ in range(args.warmup + 1):
            kda.kda_layer_prologue(*raw[:4], braw, *convs)
            kda.kda_layer_epilogue(raw[0], raw[4], nw)
    elif args.ncu_case in ("prefill", "prefill_ring", "prefill_ring_h96"):
        # prefill_ring_h96: T=8192 with K3's 96 heads, ring workspace (96 chains in groups)
        Hc = 96 if args.ncu_case == "prefill_ring_h96" else PREFILL["H"]
        x = inputs.prefill_inputs([PREFILL["T"]], H=Hc, io="bf16", seed=PREFILL["seed"],
                                  device=dev)
        kind = "fast" if args.ncu_case == "prefill" else "ring"
        ws = kda.prefill_workspace(x.q, None, N=1, T=PREFILL["T"], chunk=C, kind=kind)
        for _ in range(args.warmup + 1):
            kda.kda_prefill(x.q, x.k, x.v, x.g, x.beta, x.scale, chunk=C, workspace=ws)
    elif args.ncu_case == "decode_multi":  # T = 4 tokens per sequence through a permuted pool
        B, Hd, Tm = args.decode_batch, DECODE["H"], 4
        xm = inputs.prefill_inputs([Tm] * B, H=Hd, io="bf16", seed=DECODE["seed"] + 5, device=dev)
        shp = (B, Tm, Hd, D)
        gen = torch.Generator(device=dev)
        gen.manual_seed(DECODE["seed"] + 6)
        pool = 0.02 * torch.randn((B, Hd, D, D), generator=gen, device=dev)
        perm = torch.randperm(B, generator=gen, device=dev).to(torch.int32)
        for _ in range(args.warmup + 1):
            kda.kda_decode(xm.q.view(shp), xm.k.view(shp), xm.v.view(shp), xm.g.view(shp),
                           xm.beta.view(B, Tm, Hd), xm.scale, pool, state_indices=perm)
    else:
        q, k, v, g, beta, state, scale = inputs.decode_inputs(
            B=args.decode_batch, H=DECODE["H"], steps=1, seed=DECODE["seed"], device=dev)
        for _ in range(args.warmup + 1):
            kda.kda_decode_step(q[0], k[0], v[0], g[0], beta[0], scale, state)
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--ncu-case", choices=["prefill", "prefill_ring", "prefill_ring_h96", "decode",
                                           "decode_multi", "layer"],
                    default=None,
                    help="run only `warmup` + 1 launches of one kernel (for ncu captures)")
    ap.add_argument("--decode-batch", type=int, default=DECODE["B"])
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="the headline's timed region repeats blocks of K steps for at least this long")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the append (H=96) and varlen (64 sequences) prefill lines")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.ncu_case:
        ncu_case(args)
        return

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    import torch.distributed as dist
    import kimi_delta_attention_rule_gb300 as kda
    from kimi_delta_attention_rule_gb300 import build as kbuild, inputs

    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        kbuild.build()
    if world > 1:
        dist.barrier()
    kda.load()
    stream = torch.cuda.current_stream()

    # ---- prefill workload (each rank: its own independent batch) -----------
    x = inputs.prefill_inputs([PREFILL["T"]], H=PREFILL["H"], io="bf16",
                              seed=rank_seed(PREFILL["seed"], rank), device=dev)
    H, T = PREFILL["H"], PREFILL["T"]
    out = torch.empty_like(x.q)
    fin = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
    ws = kda.prefill_workspace(x.q, None, N=1, T=T, chunk=C)
    sched = kda.kda_prefill_schedule(1, T, H, D, C, kda.KDA_BF16)
    fused = sched == kda.KDA_SCHEDULE_FUSED
    launches_per_step = 1 if fused else 2
    kernel_label = ("kda_prefill: fused_kernel (chunk preparation and recurrence in one "
                    "cooperative launch)" if fused else
                    "kda_prefill: prep_kernel + recur_kernel (one call)")

    def step():
        kda.kda_prefill(x.q, x.k, x.v, x.g, x.beta, x.scale, cu_seqlens=None, chunk=C, out=out,
                        final_state=fin, workspace=ws, stream=stream)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(max(0, args.warmup - 3) + 2):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    est_ms = ev0.elapsed_time(ev1) / (max(0, args.warmup - 3) + 2)
    # The timed region is `blocks` blocks of exactly K steps each, enough blocks
    # for at least --min-timed-s seconds (the same count on every rank), so that
    # the clocks are sampled under load and one short window does not decide.
    blocks = max(1, math.ceil(args.min_timed_s * 1e3 / (args.steps * est_ms)))
    blocks = int(max_over_ranks(blocks, world, dev))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(blocks):
            for _ in range(args.steps):
                step()
        ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1) / (blocks * args.steps)
    ms = max_over_ranks(ms, world, dev)
    assert kda.kda_workspace_status(ws) == kda.KDA_OK
    units = H * T * world
    value = units / (ms * 1e-3) / 1e6
    clocks = clk.summary()

    # the same step with the ring-sized workspace (bounded: blocks in per-chain
    # rings instead of one per chunk)
    ring_bytes = kda.kda_prefill_workspace_size_ring(1, T, H, D, C, kda.KDA_BF16)
    bounded_ws = None
    if 0 < ring_bytes < ws.numel():
        ws_r = torch.empty(ring_bytes, dtype=torch.uint8, device=dev)
        pl = kda.kda_prefill_plan(1, T, H, D, C, kda.KDA_BF16, False, ring_bytes)
        ms_r, n_r = time_prefill_calls(
            lambda: kda.kda_prefill(x.q, x.k, x.v, x.g, x.beta, x.scale, chunk=C, out=out,
                                    final_state=fin, workspace=ws_r, stream=stream), stream)
        ms_r = max_over_ranks(ms_r, world, dev)
        assert kda.kda_workspace_status(ws_r) == kda.KDA_OK
        tr_ring = measured_traffic("prefill_ring_h32_t8192")
        bounded_ws = {"workspace_bytes": ring_bytes, "full_workspace_bytes": ws.numel(),
                      "traffic": tr_ring["bytes_per_launch"] if tr_ring else None,
                      "ms_per_call": ms_r, "calls_timed": n_r,
                      "value": H * T * world / (ms_r * 1e-3) / 1e6, "unit": "Mtok/s",
                      "vs_full_workspace": ms / ms_r,
                      "plan": {"schedule": "fused", "groups": pl.groups,
                               "group_chains": pl.group_chains, "ring": pl.ring},
                      "gpu_launches": n_r * pl.groups}
        del ws_r

    peaks, peak_src = load_peaks()
    tr_pf = measured_traffic("prefill_h32_t8192")
    if tr_pf is not None:  # DRAM bytes of one call under the schedule that ran
        kern = tr_pf["kernels"]
        names = ["fused_kernel"] if fused else ["prep_kernel (split schedule)",
                                                "recur_kernel (split schedule)"]
        tr_pf = ({"bytes_per_launch": sum(kern[k]["read"] + kern[k]["write"] for k in names)}
                 if all(k in kern for k in names) else None)
    bpt = prefill_bytes_per_head_token()
    bytes_per_launch = bpt * H * T + fin.numel() * 4
    achieved_gbs = bytes_per_launch / (ms * 1e-3) / 1e9
    flops = prefill_flops_per_chunk() * H * (T // C)
    tflops = flops / (ms * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers ---------------
    # Every step copies its inputs from pinned host memory, runs the prefill and
    # reads its output back. Consecutive steps are pipelined the way a serving
    # loop would run them: host-to-device copies on one stream, the prefill on
    # the main one, device-to-host reads on a third, with two sets of device
    # buffers, so that step i + 1's inputs and step i - 1's output cross the
    # host link while step i computes.
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv, hg, hb = pin(x.q), pin(x.k), pin(x.v), pin(x.g), pin(x.beta)
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dbufs = [[torch.empty_like(t) for t in (x.q, x.k, x.v, x.g, x.beta)] for _ in range(2)]
    douts = [out, torch.empty_like(out)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg, hb))
    d2h = hout.numel() * hout.element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer set b on the device
    ev_run = [torch.cuda.Event() for _ in range(2)]     # prefill of set b done
    ev_out = [torch.cuda.Event() for _ in range(2)]     # output of set b read back
    for b in range(2):  # all sets free at the start
        ev_run[b].record(stream)
        ev_out[b].record(stream)

    def e2e_step(i):
        b = i % 2
        dq, dk, dv, dg, db = dbufs[b]
        s_in.wait_event(ev_run[b])  # the prefill that read this set is done
        with torch.cuda.stream(s_in):
            for d_, h_ in ((dq, hq), (dk, hk), (dv, hv), (dg, hg), (db, hb)):
                d_.copy_(h_, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # this set's previous output was read back
        kda.kda_prefill(dq, dk, dv, dg, db, x.scale, chunk=C, out=douts[b], final_state=fin,
                        workspace=ws, stream=stream)
        ev_run[b].record(stream)
        s_out.wait_event(ev_run[b])
        with torch.cuda.stream(s_out):
            hout.copy_(douts[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 20))
    ev0.record(stream)
    s_in.wait_event(ev0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_out)
    ev1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = ev0.elapsed_time(ev1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_val = units / (e2e_ms * 1e-3) / 1e6
    del dbufs, douts, hq, hk, hv, hg, hb, hout

    # ---- layer prologue / epilogue on the same rows (HBM streams) ----------
    layer = None
    if not args.no_decode:
        gen = torch.Generator(device=dev)
        gen.manual_seed(PREFILL["seed"] + 11)
        raw = [torch.randn((T, H, D), generator=gen, device=dev).to(torch.bfloat16)
               for _ in range(5)]
        braw = torch.randn((T, H), generator=gen, device=dev).to(torch.bfloat16)
        convs = [0.5 * torch.randn((H, D, 4), generator=gen, device=dev) for _ in range(3)]
        nw = torch.ones(D, device=dev)
        for _ in range(3):
            lq, lk, lv, lg, lb = kda.kda_layer_prologue(*raw[:4], braw, *convs, stream=stream)
            ly = kda.kda_layer_epilogue(raw[0], raw[4], nw, stream=stream)
        torch.cuda.synchronize()
        reps_l = 50
        ev0.record(stream)
        for _ in range(reps_l):
            kda.kda_layer_prologue(*raw[:4], braw, *convs, stream=stream)
        ev1.record(stream)
        torch.cuda.synchronize()
        pro_ms = max_over_ranks(ev0.elapsed_time(ev1) / reps_l, world, dev)
        ev0.record(stream)
        for _ in range(reps_l):
            kda.kda_layer_epilogue(raw[0], raw[4], nw, y=ly, stream=stream)
        ev1.record(stream)
        torch.cuda.synchronize()
        epi_ms = max_over_ranks(ev0.elapsed_time(ev1) / reps_l, world, dev)
        rows = T * H
        pro_bytes = rows * (4 * 2 * D + 2 + 3 * 2 * D + 4 * D + 2)  # bf16 rows in, q k v g beta out
        epi_bytes = rows * 3 * 2 * D
        layer = {
            "workload": "rows of the prefill workload (T=8192, H=32, D=128), bf16, conv width 4",
            "prologue": {"ms": pro_ms, "GB/s": pro_bytes / (pro_ms * 1e-3) / 1e9,
                         "frac_hbm": pro_bytes / (pro_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                         "bytes_per_launch": pro_bytes, "kernel": "layer_prologue_kernel"},
            "epilogue": {"ms": epi_ms, "GB/s": epi_bytes / (epi_ms * 1e-3) / 1e9,
                         "frac_hbm": epi_bytes / (epi_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                         "bytes_per_launch": epi_bytes, "kernel": "layer_epilogue_kernel"},
            "gpu_launches": 2 * reps_l,
        }
        del raw, braw, convs, lq, lk, lv, lg, lb, ly

    # ---- decode: 64 steps replayed from a CUDA graph -----------------------
    decode = None
    if not args.no_decode:
        B, Hd, S = DECODE["B"], DECODE["H"], DECODE["steps"]
        dqq, dkk, dvv, dgg, dbb, state, dscale = inputs.decode_inputs(
            B=B, H=Hd, steps=S, seed=rank_seed(DECODE["seed"], rank), device=dev)
        dout = torch.empty((S, B, Hd, D), dtype=torch.bfloat16, device=dev)
        g_stream = torch.cuda.Stream()
        g_stream.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(g_stream):
            kda.kda_decode_step(dqq[0], dkk[0], dvv[0], dgg[0], dbb[0], dscale, state,
                                out=dout[0], stream=g_stream)  # warm-up launch
            g_stream.synchronize()
            with torch.cuda.graph(graph, stream=g_stream):
                for s in range(S):
                    kda.kda_decode_step(dqq[s], dkk[s], dvv[s], dgg[s], dbb[s], dscale, state,
                                        out=dout[s], stream=g_stream)
        torch.cuda.synchronize()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        reps = 5
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(g_stream)
        with torch.cuda.stream(g_stream):
            for _ in range(reps):
                graph.replay()
        e1.record(g_stream)
        torch.cuda.synchronize()
        dms = max_over_ranks(e0.elapsed_time(e1) / (reps * S), world, dev)
        state_bytes = decode_bytes_per_head_call(1) * B * Hd
        gbs = state_bytes / (dms * 1e-3) / 1e9
        decode = {
            "workload": "decode_b256_h96: B=256, H=96, D=128, 64 steps per graph, fp32 state "
                        "1.61 GB, bf16 q/k/v/beta",
            "value": gbs, "unit": "GB/s", "ms_per_step": dms,
            "tokens_per_s": B * Hd / (dms * 1e-3),
            "gflops": decode_flops_per_head_token() * B * Hd / (dms * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "traffic": decode_traffic(B * Hd),
                         "peak_source": peak_src, "kernel": "decode_kernel",
                         "algorithmic_bytes_per_launch": state_bytes},
            "gpu_launches": reps * S,
        }
        del graph, dqq, dkk, dvv, dgg, dbb, state, dout

        # multi-token decode through a state pool: T = 4 tokens per sequence,
        # pool entries addressed by a permutation (16 calls in a CUDA graph)
        Tm, calls = 4, 16
        xm = inputs.prefill_inputs([Tm] * B, H=Hd, io="bf16", seed=rank_seed(DECODE["seed"] + 5, rank),
                                   device=dev)
        shp = (B, Tm, Hd, D)
        mq, mk, mv, mg = (t.view(shp) for t in (xm.q, xm.k, xm.v, xm.g))
        mb = xm.beta.view(B, Tm, Hd)
        gen = torch.Generator(device=dev)
        gen.manual_seed(DECODE["seed"] + 6)
        pool = 0.02 * torch.randn((B, Hd, D, D), generator=gen, device=dev)
        perm = torch.randperm(B, generator=gen, device=dev).to(torch.int32)
        mout = torch.empty_like(mq)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(g_stream):
            kda.kda_decode(mq, mk, mv, mg, mb, dscale, pool, state_indices=perm, out=mout,
                           stream=g_stream)
            g_stream.synchronize()
            with torch.cuda.graph(graph, stream=g_stream):
                for _ in range(calls):
                    kda.kda_decode(mq, mk, mv, mg, mb, dscale, pool, state_indices=perm, out=mout,
                                   stream=g_stream)
        torch.cuda.synchronize()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        e0.record(g_stream)
        with torch.cuda.stream(g_stream):
            for _ in range(reps):
                graph.replay()
        e1.record(g_stream)
        torch.cuda.synchronize()
        mms = max_over_ranks(e0.elapsed_time(e1) / (reps * calls), world, dev)
        multi_bytes = decode_bytes_per_head_call(Tm) * B * Hd
        mgbs = multi_bytes / (mms * 1e-3) / 1e9
        decode["multi_token_pool"] = {
            "workload": "B=256, H=96, T=4 tokens per sequence per call, pool entries by a "
                        "permutation, 16 calls per graph",
            "value": mgbs, "unit": "GB/s", "ms_per_call": mms,
            "tokens_per_s": Tm * B * Hd / (mms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": mgbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": mgbs / peaks["hbm_gbs"],
                         "traffic": (measured_traffic("decode_multi_b256_h96_t4") or {}).get(
                             "bytes_per_launch"),
                         "peak_source": peak_src, "kernel": "decode_chunk_kernel",
                         "algorithmic_bytes_per_launch": multi_bytes},
            "gpu_launches": reps * calls,
        }
        decode["gpu_launches"] += reps * calls
        del graph, xm, mq, mk, mv, mg, mb, pool, perm, mout

    workloads = None
    if not args.no_workloads:
        workloads = bench_workloads(args, world, rank, dev, stream, peaks, peak_src)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": "Mtok/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), beta sigmoid(N), "
                "g -5*sigmoid(N))",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": T, "heads": H,
                   "parallelism": "dp%d" % world, "timed_blocks_of_K_steps": blocks,
                   "timed_steps": blocks * args.steps,
                   "l2": "inputs (%.0f MB) larger than L2; no flush" % (
                       (bpt - 2 * D) * H * T / 1e6)},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                     "traffic": (tr_pf or {}).get("bytes_per_launch"),
                     "peak_source": peak_src,
                     "kernel": kernel_label,
                     "algorithmic_bytes_per_launch": bytes_per_launch},
        "tensor": {"tflops_pages_count": tflops, "peak": peaks["bf16_tflops"],
                   "frac": tflops / peaks["bf16_tflops"],
                   "flops_per_launch": flops},
        "e2e": {"value": e2e_val, "unit": "Mtok/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": blocks * args.steps * launches_per_step,
        "clocks": clocks,
        "bounded_workspace": bounded_ws,
        "decode": decode,
        "layer": layer,
        "append": (workloads or {}).get("append"),
        "varlen": (workloads or {}).get("varlen"),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

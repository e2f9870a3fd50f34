#!/usr/bin/env python3
"""Benchmark of the attention hot path on one GB300 (or N, one process each).

One step = every row of the path on its workload:
  * 16K block-sparse causal MLA prefill: B=1, H=16, Sq=Sk=16384, Dqk=192,
    Dv=128, bf16, 256 x 512 sparse tiles, rel bias 0.01 (q - kv):
    build_block_mask -> attn_fwd -> attn_bwd (preprocess, key-parallel dK/dV
    kernel, query-parallel dQ kernel).
  * split-KV decode: B=32, H=32, Sq=1, Sk=65536, D=128, bf16, once per split
    count in {1, 2, 4, 8, 16} (partial + combine).
`value` is the prefill forward+backward throughput in TFLOP/s counting only
unmasked FLOPs (fwd 2N(Dqk+Dv), bwd 2N(3Dqk+2Dv)); decode is reported as
HBM GB/s of K+V bytes. Inputs are resident in HBM (0.34 GB prefill + 34.4 GB
decode per step, all larger than the 129 MB L2, so no flush is needed).

--impl reference times the fp64 CPU oracle (the only reference this path
has) on a bounded sample of the same workload on the host cores.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd/bwd TFLOP/s (unmasked FLOPs) & % BF16 peak; decode HBM GB/s"
PREFILL = dict(B=1, H=16, S=16384, Dqk=192, Dv=128, sparse_m=256, sparse_n=512, slope=0.01)
DECODE = dict(B=32, H=32, Sq=1, Sk=65536, D=128, splits=(1, 2, 4, 8, 16))


def causal_pairs(S):
    return S * (S + 1) // 2


def prefill_flops():
    P = PREFILL
    n = P["B"] * P["H"] * causal_pairs(P["S"])
    return 2 * n * (P["Dqk"] + P["Dv"]), 2 * n * (3 * P["Dqk"] + 2 * P["Dv"]), n


def decode_bytes():
    D = DECODE
    return D["B"] * D["H"] * D["Sk"] * D["D"] * 2 * 2  # K and V, bf16


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def file_hash(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic():
    """Per-launch DRAM bytes of each kernel from the committed ncu summary, kept
    only while the kernel source still hashes to what was profiled."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        tr = json.load(f)
    out = {}
    for name, rec in tr.items():
        try:
            if file_hash(*rec["sources"]) == rec["source_hash"]:
                out[name] = rec["bytes_per_launch"]
        except (OSError, KeyError):
            pass
    return out


class ClockSampler:
    """nvidia-smi clock / throttle samples taken during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        load = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


def reduce_max(values, world, device):
    """Max over ranks of each per-rank timing (ms): with replicas the job
    takes as long as its slowest rank. world == 1 returns the values as is."""
    if world == 1:
        return dict(values)
    import torch
    import torch.distributed as dist
    keys = sorted(values)
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return {k: float(v) for k, v in zip(keys, t.tolist())}


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (units per second)."""
    return world * units_per_rank / (ms * 1e-3)


def run_ours(args, rank, world, local_rank):
    import torch

    import block_sparse_attention_tma_gb300 as ga
    from block_sparse_attention_tma_gb300.synth import make_inputs, make_device_inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = ga.load_library()
    P, D = PREFILL, DECODE
    B, H, S, Dqk, Dv = P["B"], P["H"], P["S"], P["Dqk"], P["Dv"]
    x = make_inputs(B, H, S, S, Dqk, Dv, "bf16", seed=42 + rank)
    g = {n: t.to(dev) for n, t in x.items()}
    spec = ga.MaskSpec(kind=ga.CAUSAL, rel_bias_slope=P["slope"])
    lists = ga.alloc_block_lists(B, H, S, S, P["sparse_m"], P["sparse_n"], device=dev)
    o = torch.empty(B, H, S, Dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
    ws = torch.empty(ga.attn_bwd_workspace_bytes(torch.bfloat16, B, H, S, S, Dqk, Dv), dtype=torch.uint8,
                     device=dev)
    D = dict(DECODE, Sk=args.decode_sk)
    dx = make_device_inputs(D["B"], D["H"], D["Sq"], D["Sk"] if args.only != "prefill" else 128, D["D"], D["D"],
                            "bf16", seed=42 + rank, device=dev, dout=False)
    do_ = torch.empty(D["B"], D["H"], D["Sq"], D["D"], dtype=torch.bfloat16, device=dev)
    dlse = torch.empty(D["B"], D["H"], D["Sq"], dtype=torch.float32, device=dev)
    dws = torch.empty(max(ga.attn_fwd_splitkv_workspace_bytes(D["B"], D["H"], D["Sq"], D["D"], n)
                          for n in D["splits"]), dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    do_prefill = args.only in ("all", "prefill")
    do_decode = args.only in ("all", "decode")
    names = (["mask", "fwd", "bwd"] if do_prefill else []) + ([f"dec{n}" for n in D["splits"]] if do_decode else [])
    ev = {n: [] for n in names}
    ev_marks = []

    def step(record):
        marks = []
        if record:
            e = torch.cuda.Event(enable_timing=True)
            e.record(st)
            marks.append(e)

        def mark():
            if record:
                e = torch.cuda.Event(enable_timing=True)
                e.record(st)
                marks.append(e)

        if do_prefill:
            ga.build_block_mask(B, H, S, S, spec, lists)
            mark()
            ga.attn_fwd(g["q"], g["k"], g["v"], 0.0, spec, lists, o=o, lse=lse)
            mark()
            ga.attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, 0.0, spec, lists, dq=dq, dk=dk, dv=dv,
                        workspace=ws)
            mark()
        if do_decode:
            for n in D["splits"]:
                ga.attn_fwd_splitkv(dx["q"], dx["k"], dx["v"], 0.0, None, n, o=do_, lse=dlse, workspace=dws)
                mark()
        if record:
            ev_marks.append(marks)

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    rc = lib.gbattn_last_device_error(None)
    if rc != 0:
        raise RuntimeError(f"device error {rc} during warm-up")
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(vis.split(",")[local_rank] if vis else str(local_rank))
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(st)
    for _ in range(args.steps):
        step(True)
    t1.record(st)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    clk = clocks.stop()
    rc = lib.gbattn_last_device_error(None)
    if rc != 0:
        raise RuntimeError(f"device error {rc} in the timed region")
    for marks in ev_marks:
        for i, n in enumerate(names):
            ev[n].append(marks[i].elapsed_time(marks[i + 1]))
    per = {n: statistics.mean(v) for n, v in ev.items()}
    red = reduce_max(dict(per, total=total_ms), world, dev)
    total_ms = red.pop("total")
    per = red

    # ---------------- extensions outside the step (grouped-query paged decode)
    ext = None
    if not args.no_extensions and args.only == "all":
        ext = run_extensions(ga, torch, dev, st, rank)  # ~17 GB more beside the 34 GB decode cache
        ext.update(run_workload_sweep(ga, torch, dev, st, g, rank))

    # ---------------- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e and args.only == "all":
        e2e = run_e2e(args, ga, torch, dev, x, dx, spec, lists, st, nch=args.e2e_chunks)
    if args.only != "all":
        print(json.dumps({"only": args.only, "ms": {n: round(statistics.mean(v), 4) for n, v in ev.items()},
                          "total_ms": round(total_ms, 3)}), flush=True)
        return None

    fwd_f, bwd_f, npairs = prefill_flops()
    peaks = load_peaks()
    ms_step = total_ms / args.steps
    prefill_ms = per["mask"] + per["fwd"] + per["bwd"]
    value = job_rate(fwd_f + bwd_f, world, prefill_ms) / 1e12
    dec = {f"n={n}": round(job_rate(decode_bytes(), world, per[f"dec{n}"]) / 1e9, 1) for n in D["splits"]}
    traffic = load_traffic()
    # fwd and bwd are each timed alone (1-4 ms per launch, well short of the
    # power-capped regime the sustained figure was measured in): burst peak
    tpeak = peaks["bf16_tflops"]
    kern = {
        "attn_fwd": {"bound": "tensor", "achieved": fwd_f / (per["fwd"] * 1e-3) / 1e12, "peak": tpeak,
                     "unit": "TFLOP/s", "ms": per["fwd"], "traffic": traffic.get("attn_fwd")},
        "attn_bwd": {"bound": "tensor", "achieved": bwd_f / (per["bwd"] * 1e-3) / 1e12, "peak": tpeak,
                     "unit": "TFLOP/s", "ms": per["bwd"], "traffic": traffic.get("attn_bwd")},
    }
    best_n = min(D["splits"], key=lambda n: per[f"dec{n}"])
    kern["attn_fwd_splitkv"] = {"bound": "hbm", "achieved": decode_bytes() / (per[f"dec{best_n}"] * 1e-3) / 1e9,
                                "peak": peaks["hbm_gbs"], "unit": "GB/s", "ms": per[f"dec{best_n}"],
                                "splits": best_n, "traffic": traffic.get("attn_fwd_splitkv")}
    for k in kern.values():
        k["frac"] = round(k["achieved"] / k["peak"], 4)
        k["sm_mhz"] = clk.get("sm_mhz")
        k["peak_source"] = f"{peaks['source']} ({'burst bf16' if k['unit'] == 'TFLOP/s' else 'hbm copy'})"
        k["achieved"] = round(k["achieved"], 2)
        k["ms"] = round(k["ms"], 4)
    # dominant kernel = largest share of the step's time (decode runs once per split count)
    share = {"attn_fwd": per["fwd"], "attn_bwd": per["bwd"],
             "attn_fwd_splitkv": sum(per[f"dec{n}"] for n in D["splits"])}
    dom = max(share, key=share.get)
    roof = dict(kern[dom])
    roof["kernel"] = dom
    roof["share_of_step"] = round(share[dom] / sum(per.values()), 4)
    launches_per_step = 2 + 1 + 3 + sum(1 if n == 1 else 2 for n in D["splits"])  # lists 2, fwd 1, bwd 3
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "16K block-sparse causal MLA prefill fwd+bwd + 64K split-KV decode",
                   "prefill": "B=1 H=16 Sq=Sk=16384 Dqk=192 Dv=128 bf16 causal, sparse tiles 256x512, "
                              "kernel tiles 128x128, rel bias 0.01(q-kv)",
                   "decode": "B=32 H=32 Sq=1 Sk=65536 D=128 bf16, splits 1,2,4,8,16",
                   "parallelism": f"replicas x{world} (independent heads per rank, no collective)",
                   "l2": "inputs larger than L2 (0.34 GB prefill + 34.4 GB decode per step); no flush"},
        "fwd_tflops": round(fwd_f / (per["fwd"] * 1e-3) / 1e12, 2),
        "bwd_tflops": round(bwd_f / (per["bwd"] * 1e-3) / 1e12, 2),
        "fwd_frac_of_peak": round(fwd_f / (per["fwd"] * 1e-3) / 1e12 / tpeak, 4),
        "bwd_frac_of_peak": round(bwd_f / (per["bwd"] * 1e-3) / 1e12 / tpeak, 4),
        "decode_gbs": dec, "decode_frac_of_hbm": round(max(dec.values()) / peaks["hbm_gbs"], 4),
        "ms": {n: round(v, 4) for n, v in per.items()},
        "roofline": roof, "rooflines": kern,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    if ext is not None:
        out["extensions"] = ext
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(quick=args.quick_cpu)
    return out


def run_extensions(ga, torch, dev, st, rank, Sk=65536):
    """Grouped-query decode over a paged cache (not part of the step; timed on
    its own): B=32, H=32 query heads on Hkv=8 key/value heads, 65536 keys per
    sequence in a shuffled pool of 256-key pages, D=128, 4 splits. GB/s counts
    the unique K/V bytes (each key/value row read once per group)."""
    from block_sparse_attention_tma_gb300.synth import make_device_inputs
    B, H, Hkv, D, page, n = 32, 32, 8, 128, 256, 4
    x = make_device_inputs(B, H, 1, Sk, D, D, "bf16", seed=7 + rank, device=dev, dout=False, Hkv=Hkv)
    npg = Sk // page
    perm = torch.randperm(B * npg, generator=torch.Generator().manual_seed(11)).to(dev)
    pools = []
    for name in ("k", "v"):
        src = x[name].view(B, Hkv, npg, page, D).permute(0, 2, 1, 3, 4).reshape(B * npg, Hkv, page, D)
        pool = torch.empty_like(src)
        pool[perm] = src
        pools.append(pool)
        x[name] = None
    table = perm.view(B, npg).to(torch.int32).contiguous()
    seqlens = torch.full((B,), Sk, dtype=torch.int32, device=dev)
    o = torch.empty(B, H, 1, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, 1, dtype=torch.float32, device=dev)
    ws = torch.empty(ga.attn_fwd_splitkv_workspace_bytes(B, H, 1, D, n), dtype=torch.uint8, device=dev)
    run = lambda: ga.attn_fwd_splitkv_paged(x["q"], pools[0], pools[1], table, seqlens, 0.0, None, n,  # noqa: E731
                                            o=o, lse=lse, workspace=ws, stream=st)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    e0.record(st)
    for _ in range(reps):
        run()
    e1.record(st)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    uniq = B * Hkv * Sk * D * 2 * 2
    rc = ga.load_library().gbattn_last_device_error(None)
    if rc != 0:
        raise RuntimeError(f"device error {rc} in the extension run")
    del pools, x
    torch.cuda.empty_cache()
    return {"gqa_paged_decode": {"config": f"B={B} H={H} Hkv={Hkv} Sq=1 Sk={Sk} D={D} bf16, {page}-key pages "
                                           f"(shuffled pool), splits={n}",
                                 "ms": round(ms, 4), "unique_kv_gbs": round(uniq / (ms * 1e-3) / 1e9, 1),
                                 "kernel": "fwd_bf16_kernel<128,128> packed decode + combine"}}


def mask_pairs(kind, S, window_left=-1, block_size=0, prefix_len=0):
    """Allowed (q, k) pairs of one S x S head, from each mask's definition:
    causal j <= i; sliding i - W <= j <= i; block-diagonal i // Bs == j // Bs;
    prefix-LM j < P or j <= i."""
    if kind == "causal":
        return S * (S + 1) // 2
    if kind == "sliding":
        W = min(window_left, S - 1)
        return W * (W + 1) // 2 + (S - W) * (W + 1)
    if kind == "block_diag":
        nb, r = divmod(S, block_size)
        return nb * block_size * block_size + r * r
    if kind == "prefix_lm":
        P = min(prefix_len, S)
        return P * P + S * (S + 1) // 2 - P * (P + 1) // 2
    raise ValueError(kind)


SWEEP_TIMING = "device time per call: CUDA graph of calls each followed by a 256 MB L2 flush, flush-only graph subtracted"


def time_fwd_bwd(ga, torch, st, g, spec, lists, reps=10):
    """Device ms per call of attn_fwd and of attn_bwd. `reps` calls, each
    followed by an L2 flush (a 256 MB memset), are captured in one CUDA graph,
    replayed once to warm up and then timed with CUDA events on the capture
    stream; a graph of the flushes alone is timed the same way and
    subtracted. So neither host launch gaps (a 30 us kernel is shorter than
    a Python call) nor inputs left in L2 by the previous call enter the
    figure."""
    B, H, S, Dqk = g["q"].shape
    Dv = g["v"].shape[-1]
    dev = g["q"].device
    ga.build_block_mask(B, H, S, S, spec, lists, stream=st)
    o = torch.empty(B, H, S, Dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
    ws = torch.empty(ga.attn_bwd_workspace_bytes(torch.bfloat16, B, H, S, S, Dqk, Dv), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cs = torch.cuda.Stream(dev)
    fwd = lambda s: ga.attn_fwd(g["q"], g["k"], g["v"], 0.0, spec, lists, o=o, lse=lse, stream=s)  # noqa: E731
    bwd = lambda s: ga.attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, 0.0, spec, lists,  # noqa: E731
                                dq=dq, dk=dk, dv=dv, workspace=ws, stream=s)
    torch.cuda.synchronize()

    def graph_ms(fn):
        with torch.cuda.stream(cs):
            for _ in range(3):  # warm-up outside the capture
                if fn is not None:
                    fn(cs)
                flush.zero_()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            for _ in range(reps):
                if fn is not None:
                    fn(cs)
                flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(cs):  # a replay runs on the current stream
            graph.replay()
            torch.cuda.synchronize()
            e0.record(cs)
            graph.replay()
            e1.record(cs)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    base = graph_ms(None)
    out = [max(graph_ms(fn) - base, 0.0) / reps for fn in (fwd, bwd)]
    rc = ga.load_library().gbattn_last_device_error(None)
    if rc != 0:
        raise RuntimeError(f"device error {rc} in the workload sweep")
    return out


def sweep_masks(ga, torch, dev, st, g):
    """The other mask kinds of the 16K MLA prefill (sliding W = Sk/3,
    block-diagonal 1024, prefix-LM 2048, each with the relative bias), and the
    causal backward once more with the CTA-pair dK/dV kernel
    (gbattn_set_dkdv_cta_pair) for comparison with the default one-CTA kernel."""
    P = PREFILL
    B, H, S, Dqk, Dv = P["B"], P["H"], P["S"], P["Dqk"], P["Dv"]
    lists = ga.alloc_block_lists(B, H, S, S, P["sparse_m"], P["sparse_n"], device=dev)
    kinds = {"sliding": dict(kind=ga.SLIDING, window_left=S // 3),
             "block_diag": dict(kind=ga.BLOCK_DIAG, block_size=1024),
             "prefix_lm": dict(kind=ga.PREFIX_LM, prefix_len=2048)}
    masks = {}
    for name, kw in kinds.items():
        spec = ga.MaskSpec(rel_bias_slope=P["slope"], **kw)
        fms, bms = time_fwd_bwd(ga, torch, st, g, spec, lists)
        n = B * H * mask_pairs(name, S, window_left=kw.get("window_left", -1), block_size=kw.get("block_size", 0),
                               prefix_len=kw.get("prefix_len", 0))
        masks[name] = {"fwd_ms": round(fms, 4), "bwd_ms": round(bms, 4),
                       "fwd_tflops": round(2 * n * (Dqk + Dv) / (fms * 1e-3) / 1e12, 1),
                       "bwd_tflops": round(2 * n * (3 * Dqk + 2 * Dv) / (bms * 1e-3) / 1e12, 1)}
    spec = ga.MaskSpec(kind=ga.CAUSAL, rel_bias_slope=P["slope"])
    n = B * H * causal_pairs(S)
    prev = ga.set_dkdv_cta_pair(1)
    try:
        _, bms = time_fwd_bwd(ga, torch, st, g, spec, lists)
    finally:
        ga.set_dkdv_cta_pair(prev)
    masks["causal_cta_pair_bwd"] = {"bwd_ms": round(bms, 4),
                                    "bwd_tflops": round(2 * n * (3 * Dqk + 2 * Dv) / (bms * 1e-3) / 1e12, 1),
                                    "note": "dK/dV on CTA pairs (cta_group::2); the default one-CTA kernel is "
                                            "the bench line's attn_bwd"}
    return dict(masks, config=f"B={B} H={H} Sq=Sk={S} Dqk={Dqk} Dv={Dv} bf16, sparse tiles "
                              f"{P['sparse_m']}x{P['sparse_n']}, rel bias {P['slope']}", timing=SWEEP_TIMING)


def sweep_dense(ga, torch, dev, st, rank, reps=30):
    """The dense masked workload: B=2, H=8, S=2048, D=64, causal and causal
    sliding W=512, 128x128 lists. FLOPs count the allowed pairs."""
    from block_sparse_attention_tma_gb300.synth import make_inputs
    Bd, Hd, Sd, Dd = 2, 8, 2048, 64
    x = make_inputs(Bd, Hd, Sd, Sd, Dd, Dd, "bf16", seed=42 + rank)
    gd = {k: t.to(dev) for k, t in x.items()}
    dl = ga.alloc_block_lists(Bd, Hd, Sd, Sd, 128, 128, device=dev)
    dense = {}
    for name, kw, kind in (("causal", dict(kind=ga.CAUSAL), "causal"),
                           ("sliding_w512", dict(kind=ga.SLIDING, window_left=512), "sliding")):
        fms, bms = time_fwd_bwd(ga, torch, st, gd, ga.MaskSpec(**kw), dl, reps=reps)
        n = Bd * Hd * mask_pairs(kind, Sd, window_left=kw.get("window_left", -1))
        dense[name] = {"fwd_ms": round(fms, 4), "bwd_ms": round(bms, 4),
                       "fwd_tflops": round(2 * n * 2 * Dd / (fms * 1e-3) / 1e12, 1),
                       "bwd_tflops": round(2 * n * 5 * Dd / (bms * 1e-3) / 1e12, 1)}
    dense["config"] = f"B={Bd} H={Hd} Sq=Sk={Sd} D={Dd} bf16, kernel tiles 128x128"
    dense["timing"] = SWEEP_TIMING
    return dense


def sweep_dynamic(ga, torch, dev, st, rank, dims=(32, 64), reps=20):
    """The dynamic top-k workload: B=1, H=16, S=8192, top-2048 keys per head by
    an N(0,1) key bias, with causal; kept keys streamed compacted."""
    from block_sparse_attention_tma_gb300.synth import make_inputs
    dyn = {}
    Bd, Hd, Sd, topk = 1, 16, 8192, 2048
    for D in dims:
        x = make_inputs(Bd, Hd, Sd, Sd, D, D, "bf16", seed=42 + rank, bias=True)
        gd = {k: t.to(dev) for k, t in x.items()}
        spec = ga.MaskSpec(kind=ga.DYNAMIC_TOPK, topk=topk, key_bias=gd["key_bias"])
        dl = ga.alloc_block_lists(Bd, Hd, Sd, Sd, 128, 128, device=dev)
        fms, bms = time_fwd_bwd(ga, torch, st, gd, spec, dl, reps=reps)
        # pairs: every kept key p is seen by the rows p .. S-1
        kept = torch.topk(x["key_bias"].double(), topk, dim=-1).indices
        n = int((Sd - kept).sum())
        dyn[f"d{D}"] = {"fwd_ms": round(fms, 4), "bwd_ms": round(bms, 4),
                        "fwd_tflops": round(2 * n * 2 * D / (fms * 1e-3) / 1e12, 1),
                        "bwd_tflops": round(2 * n * 5 * D / (bms * 1e-3) / 1e12, 1)}
        del gd, dl
    dyn["config"] = (f"B={Bd} H={Hd} Sq=Sk={Sd} bf16, top-{topk} keys per head by an N(0,1) key bias, with causal; "
                     "kept keys streamed compacted")
    dyn["timing"] = SWEEP_TIMING
    return dyn


def run_workload_sweep(ga, torch, dev, st, g, rank):
    """The informational lines beside the step: the 16K MLA prefill's other
    mask kinds (and the CTA-pair dK/dV kernel), the dense masked workload and
    the dynamic top-k workload. Not part of the step; FLOPs count the allowed
    pairs (fwd 2N(Dqk+Dv), bwd 2N(3Dqk+2Dv))."""
    masks = sweep_masks(ga, torch, dev, st, g)
    dense = sweep_dense(ga, torch, dev, st, rank)
    dyn = sweep_dynamic(ga, torch, dev, st, rank)
    torch.cuda.empty_cache()
    return {"dense2k": dense, "mla16k_mask_kinds": masks, "dynamic_topk": dyn}


def run_e2e(args, ga, torch, dev, x, dx, spec, lists, st, nch=8):
    """Same step through the C ABI with host buffers: every step copies its
    inputs in from pinned host memory and its results out, inside the timed
    region. The step is cut into `nch` independent chunks (heads for the
    prefill, sequences for the decode) on `nch` streams, the way a caller of
    the stream-ordered API overlaps one chunk's copies with another's kernels;
    the work per step is the same as the device-only step."""
    P, D = PREFILL, DECODE
    B, H, S, Dqk, Dv = P["B"], P["H"], P["S"], P["Dqk"], P["Dv"]
    hc = H // nch
    streams = [torch.cuda.Stream(dev) for _ in range(nch)]
    # prefill chunk c = heads [c*hc, (c+1)*hc): contiguous host / device slices (B == 1)
    h_in = {n: t.pin_memory() for n, t in x.items()}
    outs = {"o": (B, H, S, Dv), "dq": (B, H, S, Dqk), "dk": (B, H, S, Dqk), "dv": (B, H, S, Dv)}
    h_out = {n: torch.empty(sh, dtype=torch.bfloat16).pin_memory() for n, sh in outs.items()}
    h_lse = torch.empty(B, H, S, dtype=torch.float32).pin_memory()
    chunks = []
    for c in range(nch):
        hs = slice(c * hc, (c + 1) * hc)
        ch = {"hs": hs, "in": {n: torch.empty_like(t[:, hs], device=dev) for n, t in x.items()}}
        ch["spec"] = spec
        ch["lists"] = ga.alloc_block_lists(B, hc, S, S, P["sparse_m"], P["sparse_n"], device=dev)
        ch["o"] = torch.empty(B, hc, S, Dv, dtype=torch.bfloat16, device=dev)
        ch["lse"] = torch.empty(B, hc, S, dtype=torch.float32, device=dev)
        ch["dq"] = torch.empty(B, hc, S, Dqk, dtype=torch.bfloat16, device=dev)
        ch["dk"] = torch.empty(B, hc, S, Dqk, dtype=torch.bfloat16, device=dev)
        ch["dv"] = torch.empty(B, hc, S, Dv, dtype=torch.bfloat16, device=dev)
        ch["ws"] = torch.empty(ga.attn_bwd_workspace_bytes(torch.bfloat16, B, hc, S, S, Dqk, Dv), dtype=torch.uint8,
                               device=dev)
        chunks.append(ch)
    # decode chunk c = sequences [c*bc, (c+1)*bc); the host holds the KV cache (34 GB pinned)
    bc = D["B"] // nch
    dh = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in dx.items()}
    for n, t in dx.items():
        dh[n].copy_(t)
    dd = {n: torch.empty_like(t) for n, t in dx.items()}
    d_o = torch.empty(D["B"], D["H"], D["Sq"], D["D"], dtype=torch.bfloat16, device=dev)
    d_lse = torch.empty(D["B"], D["H"], D["Sq"], dtype=torch.float32, device=dev)
    h_do = torch.empty(d_o.shape, dtype=torch.bfloat16).pin_memory()
    nmax = max(D["splits"])
    dws = [torch.empty(ga.attn_fwd_splitkv_workspace_bytes(bc, D["H"], D["Sq"], D["D"], nmax), dtype=torch.uint8,
                       device=dev) for _ in range(nch)]

    def prefill():
        for ch, s in zip(chunks, streams):
            hs = ch["hs"]
            with torch.cuda.stream(s):
                for n in h_in:
                    ch["in"][n].copy_(h_in[n][:, hs], non_blocking=True)
                sp = ga.MaskSpec(kind=spec.kind, rel_bias_slope=spec.rel_bias_slope)
                ga.build_block_mask(B, hc, S, S, sp, ch["lists"])
                ga.attn_fwd(ch["in"]["q"], ch["in"]["k"], ch["in"]["v"], 0.0, sp, ch["lists"], o=ch["o"],
                            lse=ch["lse"])
                ga.attn_bwd(ch["in"]["q"], ch["in"]["k"], ch["in"]["v"], ch["o"], ch["in"]["do"], ch["lse"], 0.0,
                            sp, ch["lists"], dq=ch["dq"], dk=ch["dk"], dv=ch["dv"], workspace=ch["ws"])
                for n in ("o", "dq", "dk", "dv"):
                    h_out[n][:, hs].copy_(ch[n], non_blocking=True)
                h_lse[:, hs].copy_(ch["lse"], non_blocking=True)

    def decode():
        for c, s in enumerate(streams):
            bs = slice(c * bc, (c + 1) * bc)
            with torch.cuda.stream(s):
                for n in dh:
                    dd[n][bs].copy_(dh[n][bs], non_blocking=True)
                ga.attn_fwd_splitkv(dd["q"][bs], dd["k"][bs], dd["v"][bs], 0.0, None, nmax, o=d_o[bs], lse=d_lse[bs],
                                    workspace=dws[c])
                h_do[bs].copy_(d_o[bs], non_blocking=True)

    steps = max(2, min(args.steps, 5))
    res = {}
    for name, fn in (("prefill", prefill), ("decode", decode)):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            fn()
        torch.cuda.synchronize()
        res[name] = (time.perf_counter() - t0) / steps
    rc = ga.load_library().gbattn_last_device_error(None)
    if rc != 0:
        raise RuntimeError(f"device error {rc} in the end-to-end run")
    fwd_f, bwd_f, _ = prefill_flops()
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values()) + h_lse.numel() * 4
    dh2d = sum(t.numel() * t.element_size() for t in dh.values())
    return {"value": round((fwd_f + bwd_f) / res["prefill"] / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(res["prefill"] * 1e3, 3),
            "pipelining": f"{nch} head chunks (prefill) / {nch} sequence chunks (decode) on {nch} streams",
            "decode": {"value": round(decode_bytes() / res["decode"] / 1e9, 1), "unit": "GB/s",
                       "splits": nmax, "h2d_bytes_per_step": dh2d,
                       "d2h_bytes_per_step": h_do.numel() * 2, "ms_per_step": round(res["decode"] * 1e3, 3)},
            "steps": steps}


def cpu_baseline(quick=False):
    """The fp64 oracle on a bounded sample: one (b, h) head of the prefill
    workload (forward + backward) and one head of the decode workload."""
    import numpy as np
    import torch

    from block_sparse_attention_tma_gb300.synth import make_inputs
    from oracle import attention as orc

    P = PREFILL
    S = 4096 if quick else P["S"]
    x = make_inputs(1, 1, S, S, P["Dqk"], P["Dv"], "bf16", seed=42)
    f = {n: t.float().double().numpy()[0, 0] for n, t in x.items()}
    prob = orc.Problem(f["q"], f["k"], f["v"], kind=orc.CAUSAL, rel_bias_slope=P["slope"])
    t0 = time.perf_counter()
    prob.forward()
    t1 = time.perf_counter()
    prob.backward(f["do"])
    t2 = time.perf_counter()
    n = causal_pairs(S)
    flops = 2 * n * (P["Dqk"] + P["Dv"]) + 2 * n * (3 * P["Dqk"] + 2 * P["Dv"])
    D = DECODE
    g = torch.Generator().manual_seed(42)
    q = torch.randn(1, D["D"], generator=g).bfloat16().double().numpy()
    k = torch.randn(D["Sk"], D["D"], generator=g).bfloat16().double().numpy()
    v = torch.randn(D["Sk"], D["D"], generator=g).bfloat16().double().numpy()
    t3 = time.perf_counter()
    orc.Problem(q, k, v).forward()
    t4 = time.perf_counter()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(flops / (t2 - t0) / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"prefill: one (b,h) head, Sq=Sk={S}, causal, rel bias, fwd+bwd in fp64 "
                      f"({(t2 - t0):.1f} s); decode: one head, Sk={D['Sk']} ({(t4 - t3) * 1e3:.0f} ms)",
            "fwd_s": round(t1 - t0, 2), "bwd_s": round(t2 - t1, 2),
            "decode_gbs": round(D["Sk"] * D["D"] * 2 * 2 / (t4 - t3) / 1e9, 3)}


def run_reference(args):
    """The fp64 oracle, as it stands, on the host cores; each step is one
    bounded sample of the prefill workload (one head, forward + backward)."""
    import numpy as np  # noqa: F401

    from block_sparse_attention_tma_gb300.synth import make_inputs
    from oracle import attention as orc

    P = PREFILL
    S = args.ref_seq
    x = make_inputs(1, 1, S, S, P["Dqk"], P["Dv"], "bf16", seed=42)
    f = {n: t.float().double().numpy()[0, 0] for n, t in x.items()}
    prob = orc.Problem(f["q"], f["k"], f["v"], kind=orc.CAUSAL, rel_bias_slope=P["slope"])
    n = causal_pairs(S)
    flops = 2 * n * (P["Dqk"] + P["Dv"]) + 2 * n * (3 * P["Dqk"] + 2 * P["Dv"])
    for _ in range(args.warmup):
        prob.forward()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        prob.forward()
        prob.backward(f["do"])
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = flops / (ms * 1e-3) / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = f"one (b,h) head of the 16K causal MLA prefill at Sq=Sk={S}, fwd+bwd, fp64"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "16K block-sparse causal MLA prefill fwd+bwd (oracle sample)", "sample": sample},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=8, choices=[1, 2, 4, 8, 16],
                    help="independent chunks (and streams) of the end-to-end step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extensions", action="store_true", help="skip the informational lines (paged GQA decode, mask-kind and dynamic sweeps)")
    ap.add_argument("--quick-cpu", action="store_true", help="cpu_baseline on a 4096-token sample")
    ap.add_argument("--ref-seq", type=int, default=4096, help="sequence length of the reference-arm sample")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "gqa", "dense2k", "dynamic"], default="all",
                    help="time one part only (profiling runs); prints a short line, not the bench line")
    ap.add_argument("--dyn-d", type=int, default=0, help="head dim of the dynamic workload (--only dynamic; 0 = 32 and 64)")
    ap.add_argument("--gqa-sk", type=int, default=65536, help="keys of the grouped-query decode (--only gqa)")
    ap.add_argument("--decode-sk", type=int, default=DECODE["Sk"], help="decode keys (profiling runs only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.only == "all" and args.decode_sk != DECODE["Sk"]:
        ap.error("--decode-sk is for profiling runs with --only")
    if args.only in ("gqa", "dense2k", "dynamic"):
        import torch
        import block_sparse_attention_tma_gb300 as ga
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        st = torch.cuda.current_stream(dev)
        if args.only == "gqa":
            ext = run_extensions(ga, torch, dev, st, rank, Sk=args.gqa_sk)
        elif args.only == "dense2k":
            ext = {"dense2k": sweep_dense(ga, torch, dev, st, rank, reps=max(args.steps, 30))}
        else:
            ext = {"dynamic_topk": sweep_dynamic(ga, torch, dev, st, rank, dims=(args.dyn_d,) if args.dyn_d else (32, 64),
                                                 reps=max(args.steps, 20))}
        if rank == 0:
            print(json.dumps({"only": args.only, **ext}), flush=True)
    else:
        out = run_ours(args, rank, world, local_rank)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

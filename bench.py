#!/usr/bin/env python
"""Benchmark of the DSA sparse-attention hot path on one node.

Default workload: batched decode (32 requests, kv_len ~ U{4096..8192}, pool of
8192 pages, token top-k k=2048, 128-head absorbed-MLA attention). One step =
indexer score + exact token top-k + sparse MLA decode over the whole batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0. ``--impl reference`` times the CPU oracle (the
only reference this path has) on a bounded sample of the same workload.
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the path
has no exchange step; ranks only meet for the timing barrier and the max.
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "DSA layer tokens/s (decode, prefill) and % of HBM / tensor-core roofline"

# the key lengths of each workload, as the dsa_inputs builders draw them
KV_LEN_DESC = {
    "tiny_decode": "1024",
    "batched_decode": "U{4096..8192}",
    "long_decode": "131072",
    "single_prefill": "8192 (one request, prefix 0)",
    "ragged_mixed": "decode U{8192..131072}; extends of 4096 on prefixes 0/16384/65536/110592",
}

L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="batched_decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(seconds, world):
    """The slowest rank's time (replicas are timed independently; the job
    takes as long as its slowest replica). Uses the default process group."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as tdist

    t = torch.tensor([seconds], dtype=torch.float64)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_step, steps, world, seconds):
    """Whole-job tokens/s of ``world`` replicas that each ran ``steps`` steps
    of ``tokens_per_step`` tokens in at most ``seconds``."""
    return tokens_per_step * steps * world / seconds


# ----------------------------------------------------------------- helpers
def blas_threads():
    """Threads of the BLAS numpy runs the oracle's matmuls on."""
    try:
        with open("/proc/self/maps") as f:
            libs = {l.split()[-1] for l in f if "openblas" in l.lower() and l.split()[-1].startswith("/")}
        for path in libs:
            lib = ctypes.CDLL(path)
            for fn in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                       "openblas_get_num_threads", "scipy_openblas_get_num_threads"):
                if hasattr(lib, fn):
                    return int(getattr(lib, fn)())
    except Exception:
        pass
    return os.cpu_count() or 1


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for l in self.lines:
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append((float(p[1]), float(p[2]), p[5], p[6], p[7], p[8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 peak: the burst figure, since stages are timed alone."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["bf16_tflops"], "measured (burst)"
    except Exception:
        return 1900.0, "fallback"


def committed_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, only while the
    kernel source is unchanged since the counters were taken."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)[kernel_key]
        src = os.path.join(ROOT, d["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return d["bytes_per_launch"] if h == d["source_sha256_16"] else None
    except Exception:
        return None


def stage_roofline(wl, rn, timed):
    """Time every stage of one layer in isolation (L2 flushed before each)
    and set its algorithmic work against the roofline it is bound by:
    decode indexer 256 B per visible key and decode attention 1152 B per
    selected visible key (HBM); prefill indexer 2*32*128 FLOP per visible
    (query, key) pair and query-block attention 2*H*(576+512) FLOP per
    (query, selected visible key) pair (tensor, bf16). The paged write-back
    that precedes the path is timed beside them (not part of the step):
    2 B read + 2 B written per copied element (HBM)."""
    import numpy as np
    import torch

    rg = wl.rg
    hbm, hbm_kind = measured_peaks()
    tfl, tfl_kind = measured_tensor_peak()
    nvis = np.clip(np.minimum(rg.seq_lens[rg.token_seq()], rg.token_pos() + 1), 0, None).astype(np.int64)
    out = {}

    def entry(ms, work, bound):
        if bound == "hbm":
            ach = work / (ms * 1e-3) / 1e9
            return {"ms": ms, "algorithmic_bytes": int(work), "bound": "hbm", "achieved": ach, "unit": "GB/s",
                    "peak": hbm, "peak_kind": hbm_kind, "frac": ach / hbm}
        ach = work / (ms * 1e-3) / 1e12
        return {"ms": ms, "algorithmic_flops": int(work), "bound": "tensor", "achieved": ach, "unit": "TFLOP/s",
                "peak": tfl, "peak_kind": tfl_kind, "frac": ach / tfl}

    ps = rg.page_size
    if rn.prefill or rn.page_budget is not None:
        tp = rn.topk_pages[0].cpu().numpy().astype(np.int64)
        keys = np.where(tp >= 0, np.clip(nvis[:, None] - tp * ps, 0, ps), 0).sum()
    else:
        keys = int((rn.topk[0] >= 0).sum().item())
    if rn.prefill:
        out["indexer_page_topk"] = entry(timed(lambda: rn.index(0)), 2 * 32 * 128 * nvis.sum(), "tensor")
        out["block_union"] = entry(timed(lambda: rn.union(0)), rn.topk_pages[0].numel() * 4, "hbm")
        out["sparse_mla_prefill_qblock"] = entry(timed(lambda: rn.attend(0)), 2 * wl.H * (576 + 512) * keys,
                                                 "tensor")
    else:
        name = "indexer_page_topk" if rn.page_budget is not None else "indexer_topk"
        out[name] = entry(timed(lambda: rn.index(0)), 256 * nvis.sum(), "hbm")
        out["sparse_mla_decode"] = entry(timed(lambda: rn.attend(0)), 1152 * keys, "hbm")
    # the step before the path: paged write-back of every query token's
    # latent row and indexer key (the rows already there are written back
    # unchanged, so the caches keep their contents): 2 x (576 + 128) x 2 B per
    # token, read and written
    import deepseek_sparse_attention_score_gb300 as dsa

    tseq, tpos = rg.token_seq(), rg.token_pos()
    ent = rg.cu_kv_lens[tseq] // ps + tpos // ps
    phys = torch.from_numpy((rg.page_indices[ent].astype(np.int64) * ps + tpos % ps)).to(rn.kv[0].device)
    kv_rows = rn.kv[0].view(-1, rn.kv[0].shape[-1]).index_select(0, phys)[:, :576].contiguous()
    k_rows = rn.kcache[0].view(-1, 128).index_select(0, phys).contiguous()

    def write_back():
        dsa.dsa_paged_write_back(kv_rows, rn.kv[0], *rn.meta, D=576, dev_status=rn.status)
        dsa.dsa_paged_write_back(k_rows, rn.kcache[0], *rn.meta, D=128, dev_status=rn.status)

    out["paged_write_back"] = entry(timed(write_back), 2 * (576 + 128) * 2 * rg.T, "hbm")
    out["paged_write_back"]["in_step"] = False
    # the dense fallback (layers without an indexer) over the same queries:
    # every visible position, 1152 B (decode, HBM) or 2*H*(576+512) FLOP
    # (prefill, tensor) per visible (query, key) pair; timed beside the step
    if args_workload_allows_dense(wl):
        o_dense = torch.empty_like(rn.o[0])
        ws_dense = torch.empty(max(1, dsa.dsa_sparse_mla_decode_workspace_size(rg.T, wl.H)), dtype=torch.uint8,
                               device=rn.kv[0].device)

        def dense():
            dsa.dsa_dense_mla(rn.q[0], rn.kv[0], *rn.meta, max_kv=int(rg.seq_lens.max()), sm_scale=wl.sm_scale,
                              o=o_dense, ws=ws_dense, dev_status=rn.status)

        pairs = int(nvis.sum())
        if rn.prefill:
            out["dense_mla"] = entry(timed(dense, reps=3), 2 * wl.H * (576 + 512) * pairs, "tensor")
        else:
            out["dense_mla"] = entry(timed(dense), 1152 * pairs, "hbm")
        out["dense_mla"]["in_step"] = False
    # the approximate top-k (the pages' fast-path trade) on the decode rows,
    # with its recall against the exact selection of the step
    if not rn.prefill and rn.page_budget is None:
        over = 4
        ws_ap = torch.empty(max(1, dsa.lib().dsa_indexer_topk_approx_workspace_size(
            rg.T, rg.S, int(rg.seq_lens.max()), ps, wl.k, over)), dtype=torch.uint8, device=rn.kv[0].device)
        sel_ap = torch.empty((rg.T, wl.k), dtype=torch.int32, device=rn.kv[0].device)

        def approx():
            dsa.dsa_indexer_topk_approx(rn.q_idx, rn.w, rn.kcache[0], *rn.meta, k=wl.k, max_kv=int(rg.seq_lens.max()),
                                        over=over, topk=sel_ap, ws=ws_ap, dev_status=rn.status)

        e = entry(timed(approx), 256 * nvis.sum(), "hbm")
        a, x = sel_ap.cpu().numpy(), rn.topk[0].cpu().numpy()
        hit = sum(len(np.intersect1d(a[t][a[t] >= 0], x[t][x[t] >= 0])) for t in range(rg.T))
        e["recall_vs_exact"] = hit / max(1, int((x >= 0).sum()))
        e["over"] = over
        e["in_step"] = False
        out["indexer_topk_approx"] = e
    return out


def args_workload_allows_dense(wl):
    """The dense fallback is timed on the single-layer workloads (the mixed
    four-layer batch would take seconds per call)."""
    return wl.name in ("tiny_decode", "batched_decode", "long_decode", "single_prefill")


# ---------------------------------------------------------------- oracle leg
def host_sample(wl, seqs, layer=0):
    """Compact CPU copy of the requests ``seqs`` of a workload: their query
    tokens and only their own pages (renumbered), for the CPU oracle."""
    import numpy as np
    import torch

    rg = wl.rg
    ps = rg.page_size
    pages, pi, cu_kv, toks = [], [], [0], []
    for s in seqs:
        npg = -(-int(rg.seq_lens[s]) // ps)
        b = int(rg.cu_kv_lens[s]) // ps
        pi.extend(range(len(pages), len(pages) + npg))
        pages.extend(rg.page_indices[b:b + npg].tolist())
        cu_kv.append(cu_kv[-1] + npg * ps)
        toks.extend(range(int(rg.cu_q_lens[s]), int(rg.cu_q_lens[s + 1])))
    dev = wl.kcache[0].device
    pidx = torch.tensor(pages, dtype=torch.long, device=dev)
    tidx = torch.tensor(toks, dtype=torch.long, device=dev)
    f = lambda t: t.float().cpu().numpy()
    q_lens = np.diff(rg.cu_q_lens)[list(seqs)]
    return dict(
        q_idx=f(wl.q_idx.to(dev)[tidx]), w=f(wl.w.to(dev)[tidx]), kcache=f(wl.kcache[0][pidx]),
        q=f(wl.q[layer].to(dev)[tidx]), kv=f(wl.kv[layer][pidx]),
        seq_lens=rg.seq_lens[list(seqs)].copy(),
        cu_q_lens=np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32),
        cu_kv_lens=np.asarray(cu_kv, np.int32), page_indices=np.asarray(pi, np.int32), ntok=len(toks))


def oracle_decode_step(smp, k, sm_scale):
    import oracle as O

    meta = dict(seq_lens=smp["seq_lens"], cu_q_lens=smp["cu_q_lens"], cu_kv_lens=smp["cu_kv_lens"],
                page_indices=smp["page_indices"])
    topk, _ = O.indexer_topk(smp["q_idx"], smp["w"], smp["kcache"], k=k, **meta)
    o, _ = O.sparse_mla(smp["q"], smp["kv"], sel=topk, unit=1, sm_scale=sm_scale, Dv=512, **meta)
    return o


def time_oracle(wl, min_seconds=10.0, max_seconds=30.0):
    """Oracle throughput on a bounded sample: requests are taken one at a
    time, in order (wrapping around), until at least ``min_seconds`` of CPU
    work has been timed."""
    total, toks, nreq = 0.0, 0, 0
    S = wl.rg.S
    while total < min_seconds and total < max_seconds:
        smp = host_sample(wl, [nreq % S])
        t0 = time.perf_counter()
        oracle_decode_step(smp, wl.k, wl.sm_scale)
        total += time.perf_counter() - t0
        toks += smp["ntok"]
        nreq += 1
    return toks / total, total, toks, nreq


# --------------------------------------------------------------- reference
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import dsa_inputs as DI

    wl = DI.WORKLOADS[args.workload]()
    S = wl.rg.S
    cores = blas_threads()
    times, toks = [], 0
    for i in range(args.warmup + args.steps):
        s = i % S
        smp = host_sample(wl, [s])
        t0 = time.perf_counter()
        oracle_decode_step(smp, wl.k, wl.sm_scale)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            toks += smp["ntok"]
    total = sum(times)
    value = toks / total
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, "sample": "one request (its decode token) per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} requests of the {args.workload} workload, one per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- ours
def run_ours(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as tdist

        tdist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as dsa
    import dsa_inputs as DI
    from deepseek_sparse_attention_score_gb300.layer import LayerRunner

    wl = DI.WORKLOADS[args.workload](device=dev)
    rn = LayerRunner(wl, dev)
    T = rn.T
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # eager warm-up (also sets kernel attributes) and launches per step
    for _ in range(max(1, args.warmup)):
        rn.step()
    torch.cuda.synchronize()
    c0 = dsa.dsa_launch_count()
    rn.step()
    torch.cuda.synchronize()
    launches_per_step = dsa.dsa_launch_count() - c0
    assert rn.status.item() == 0, f"device status {rn.status.item():#x}"

    # CUDA graph of one step (launch overhead of the ~6 small kernels removed)
    graph = None
    try:
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                rn.step()
        torch.cuda.current_stream(dev).wait_stream(s)
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        graph = g
    except Exception as e:  # pragma: no cover - reported in the JSON line
        graph_err = repr(e)[:200]
    run = graph.replay if graph is not None else rn.step

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        # keep the GPU busy with back-to-back steps for ~1.5 s around the timed
        # steps so the 200 ms clock samples land under the same load
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            for _ in range(20):
                flush.zero_()
                run()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record()
            run()
            ends[i].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - w0
        barrier()
        t_end = time.perf_counter() + 0.5
        while time.perf_counter() < t_end:
            for _ in range(20):
                flush.zero_()
                run()
            torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    value = replica_throughput(T, args.steps, world, total_s)
    clocks = clk.summary()

    # per-ABI-call times (eager, L2 flushed before each) for the roofline
    def timed(fn, reps=10):
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    kern = stage_roofline(wl, rn, timed)
    dom = max((k for k in kern if kern[k].get("in_step", True)), key=lambda k: kern[k]["ms"])
    d = kern[dom]
    roof = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"], "unit": d["unit"],
            "frac": d["frac"], "peak_kind": d["peak_kind"], "traffic": committed_traffic(dom)}

    # end to end through the public API with host buffers
    pin = lambda t: t.detach().to("cpu").pin_memory()
    h_q_idx, h_w = pin(rn.q_idx), pin(rn.w)
    h_q = [pin(x) for x in rn.q]
    h_meta = [pin(m) for m in rn.meta]
    h_topk = torch.empty(rn.topk[0].shape, dtype=torch.int32).pin_memory()
    h_o = [torch.empty(x.shape, dtype=torch.bfloat16).pin_memory() for x in rn.o]
    h2d = sum(t.numel() * t.element_size() for t in [h_q_idx, h_w, *h_q, *h_meta])
    d2h = h_topk.numel() * 4 + sum(x.numel() * 2 for x in h_o)

    # the whole host-buffer step (copies on two streams, kernels) as one
    # CUDA graph; every replay copies the inputs in and the outputs out
    side = torch.cuda.Stream(dev)
    e2e_eager = lambda: rn.step_host(h_q_idx, h_w, h_q, h_meta, h_topk, h_o, side)
    e2e_step, e2e_graph = e2e_eager, False
    try:
        s2 = torch.cuda.Stream(dev)
        s2.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s2):
            e2e_eager()  # warm the host-side caches before capture
        torch.cuda.current_stream().wait_stream(s2)
        torch.cuda.synchronize()
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=s2):
            e2e_eager()
        torch.cuda.synchronize()
        e2e_step, e2e_graph = g2.replay, True
    except Exception:  # capture unsupported here: time the eager call
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        e2e_step()
        b.record()
        torch.cuda.synchronize()
        e_ms.append(a.elapsed_time(b))
    e2e_s = max_over_ranks(sum(e_ms) / 1e3, world)
    e2e = {"value": replica_throughput(T, args.steps, world, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * e2e_s / args.steps, "cuda_graph": e2e_graph}

    cpu = None
    decode_workload = not rn.prefill and rn.page_budget is None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and decode_workload:
        v, dt, ntok, nreq = time_oracle(wl)
        cpu = {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"{nreq} requests of the {args.workload} workload taken in order ({ntok} decode "
                         f"tokens: indexer + top-k + sparse MLA), {dt:.1f} s of CPU time"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "requests": wl.rg.S, "tokens_per_step": T,
                       "layers": len(rn.types),
                       "kv_len": KV_LEN_DESC.get(args.workload, "per request, from the workload"),
                       "k": wl.k, "mla_heads": wl.H, "page_size": wl.rg.page_size,
                       "l2": "flushed (512 MB write) before every timed step", "cuda_graph": graph is not None,
                       "parallelism": "replicas" if world > 1 else "single"},
            "roofline": roof, "kernels": kern, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
            "clocks": clocks, "clock_window": "1.5 s of back-to-back steps enclosing the timed steps",
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

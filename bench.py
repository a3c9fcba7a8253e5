#!/usr/bin/env python
"""Benchmark of the DSA sparse-attention hot path on one node.

Default workload: the ragged mixed batch (48 decode tokens with kv_len
~ U{8192..131072} plus 4 chunked-prefill extends of 4096 tokens on prefixes
0/16384/65536/110592; four layers [full, shared, shared, full] with
IndexShare; token top-k k=2048 and 32-page top-k; query blocks of 256 over
the block unions; 128-head absorbed-MLA attention). One step = every layer of
the workload once: on full layers the indexer score + token top-k + page
top-k + block union, and the sparse MLA attention on every layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--only] [--no-cpu-baseline]

Prints ONE JSON line on rank 0. Beside the headline workload the line carries
per-stage numbers of the batched decode, long-context decode and single
prefill workloads (``workloads``; skipped with ``--only``).
``--impl reference`` times the CPU oracle (the only reference this path has)
on a bounded row sample of the same workload. Multi-GPU runs (torchrun, one
rank per GPU) are independent replicas: the path has no exchange step; ranks
only meet for the timing barrier and the max.
"""
from __future__ import annotations

import argparse
import json
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
# workloads whose stages ride along in the headline line
SIDE_WORKLOADS = ("batched_decode", "long_decode", "single_prefill")

L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2
MLA_DK, MLA_DV, IDX_FLOP_PER_PAIR = 576, 512, 2 * 32 * 128


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ragged_mixed")
    ap.add_argument("--only", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


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


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


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


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return None


def measured_peaks():
    d = _peaks()
    return (d["hbm_gbs"], "measured") if d else (6800.0, "fallback")


def measured_tensor_peak():
    """Dense bf16 peak: the burst figure, since stages are timed alone."""
    d = _peaks()
    return (d["bf16_tflops"], "measured (burst)") if d else (1900.0, "fallback")


def committed_traffic(kernel_key, workload):
    """DRAM bytes per launch from a committed ncu summary, only for the same
    workload and while the kernel source is unchanged since the counters were
    taken."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)[f"{kernel_key}@{workload}"]
        for src, want in d["sources"].items():
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest()[:16] != want:
                    return None
        return d["bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------ work per row
def row_work(wl, prefill, page_budget=None):
    """Per query token: visible keys (the indexer's score pairs) and the keys
    its attention reads (the selection size, capped by what is visible)."""
    import numpy as np

    rg = wl.rg
    nvis = np.clip(np.minimum(rg.seq_lens[rg.token_seq()], rg.token_pos() + 1), 0, None).astype(np.int64)
    if prefill or page_budget is not None:
        cap = (page_budget or wl.k_pages) * rg.page_size
    else:
        cap = wl.k
    return nvis, np.minimum(nvis, cap)


# ------------------------------------------------------------- GPU stages
def stage_roofline(wl, rn, timed, extras=True):
    """Time every stage of one layer in isolation (L2 flushed before each)
    and set its algorithmic work against the roofline it is bound by:
    decode indexer 256 B per visible key and decode attention 1152 B per
    selected visible key (HBM); prefill indexer 2*32*128 FLOP per visible
    (query, key) pair and query-block attention 2*H*(576+512) FLOP per
    (query, selected visible key) pair (tensor, bf16). ``per_step`` is how
    many times the stage runs in one step. With ``extras`` the calls timed
    beside the step follow: the paged write-back, the dense fallback and the
    approximate top-k."""
    import numpy as np
    import torch

    rg = wl.rg
    hbm, hbm_kind = measured_peaks()
    tfl, tfl_kind = measured_tensor_peak()
    nvis, _ = row_work(wl, rn.prefill, rn.page_budget)
    out = {}
    n_layers, n_full = len(rn.types), rn.num_full

    def entry(ms, work, bound, per_step=1):
        if bound == "hbm":
            ach = work / (ms * 1e-3) / 1e9
            return {"ms": ms, "per_step": per_step, "algorithmic_bytes": int(work), "bound": "hbm",
                    "achieved": ach, "unit": "GB/s", "peak": hbm, "peak_kind": hbm_kind, "frac": ach / hbm}
        ach = work / (ms * 1e-3) / 1e12
        return {"ms": ms, "per_step": per_step, "algorithmic_flops": int(work), "bound": "tensor",
                "achieved": ach, "unit": "TFLOP/s", "peak": tfl, "peak_kind": tfl_kind, "frac": ach / tfl}

    ps = rg.page_size
    if rn.prefill or rn.page_budget is not None:
        tp = rn.topk_pages[0].cpu().numpy().astype(np.int64)
        keys = np.where(tp >= 0, np.clip(nvis[:, None] - tp * ps, 0, ps), 0).sum()
    else:
        keys = int((rn.topk[0] >= 0).sum().item())
    if rn.prefill:
        out["indexer_page_topk"] = entry(timed(lambda: rn.index(0)), IDX_FLOP_PER_PAIR * nvis.sum(), "tensor",
                                         n_full)
        out["block_union"] = entry(timed(lambda: rn.union(0)), rn.topk_pages[0].numel() * 4, "hbm", n_full)
        out["sparse_mla_prefill_qblock"] = entry(timed(lambda: rn.attend(0)),
                                                 2 * wl.H * (MLA_DK + MLA_DV) * keys, "tensor", n_layers)
    else:
        name = "indexer_page_topk" if rn.page_budget is not None else "indexer_topk"
        out[name] = entry(timed(lambda: rn.index(0)), 256 * nvis.sum(), "hbm", n_full)
        out["sparse_mla_decode"] = entry(timed(lambda: rn.attend(0)), 1152 * keys, "hbm", n_layers)
    if not extras:
        return out
    # the first stage of every layer: paged write-back of the new tokens'
    # latent rows and (full layers) indexer keys (the synthetic caches already
    # hold these rows, so they are written back unchanged): 2 x (576 + 128) x
    # 2 B per token, read and written, on a full layer
    import deepseek_sparse_attention_score_gb300 as dsa

    out["paged_write_back"] = entry(timed(lambda: rn.write_back(0)), 2 * (576 + 128) * 2 * rg.T, "hbm", n_layers)
    # the dense fallback (layers without an indexer) over the same queries:
    # every visible position, 1152 B (decode, HBM) or 2*H*(576+512) FLOP
    # (prefill, tensor) per visible (query, key) pair; timed beside the step
    if wl.name in ("tiny_decode", "batched_decode", "long_decode", "single_prefill"):
        o_dense = torch.empty_like(rn.o[0])
        ws_dense = torch.empty(max(1, dsa.dsa_sparse_mla_decode_workspace_size(rg.T, wl.H)), dtype=torch.uint8,
                               device=rn.kv[0].device)

        def dense():
            dsa.dsa_dense_mla(rn.q[0], rn.kv[0], *rn.meta, max_kv=int(rg.seq_lens.max()), sm_scale=wl.sm_scale,
                              o=o_dense, ws=ws_dense, dev_status=rn.status)

        pairs = int(nvis.sum())
        if rn.prefill:
            out["dense_mla"] = entry(timed(dense, reps=3), 2 * wl.H * (MLA_DK + MLA_DV) * pairs, "tensor")
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


def dominant_stage(kern):
    """The in-step stage with the most time per step (time x runs per step)."""
    return max((k for k in kern if kern[k].get("in_step", True)), key=lambda k: kern[k]["ms"] * kern[k]["per_step"])


# ---------------------------------------------------------------- oracle leg
def sample_tokens(wl, n_rows, seed):
    """A stratified row sample: a third of the rows from the single-token
    (decode) requests, the rest spread evenly over the multi-token requests,
    uniformly at random inside each group (seeded)."""
    import numpy as np

    rg = wl.rg
    rng = np.random.default_rng(seed)
    ql = rg.q_lens
    dec = np.array([int(rg.cu_q_lens[s]) for s in range(rg.S) if ql[s] == 1], np.int64)
    multi = [s for s in range(rg.S) if ql[s] > 1]
    n_dec = n_rows if not multi else (min(len(dec), max(1, n_rows // 3)) if len(dec) else 0)
    picks = list(rng.choice(dec, size=min(len(dec), n_dec), replace=False)) if len(dec) else []
    if multi:
        per = max(1, (n_rows - len(picks)) // len(multi))
        for s in multi:
            t0 = int(rg.cu_q_lens[s])
            picks += list(t0 + rng.choice(int(ql[s]), size=min(int(ql[s]), per), replace=False))
    return sorted(int(t) for t in picks)


def _host_bits(t):
    """bf16 tensor -> uint16 numpy bit patterns (exact, half the bytes of fp32);
    fp32 tensors stay fp32."""
    import torch

    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view("uint16")
    return t.float().cpu().numpy()


def oracle_sample_seconds(wl, tokens, prefill, page_budget=None):
    """Oracle time of one step (every layer of the workload) over the sampled
    rows ``tokens``: per full layer the indexer score + token top-k (+ page
    top-k), per layer the sparse MLA attention over the row's selection (page
    units on the prefill path: the per-query form, which the oracle pins equal
    to the query-block form). Host copies of the rows and pages the sample
    touches are made outside the timed calls. Returns the seconds."""
    import numpy as np
    import torch

    import oracle as O

    rg = wl.rg
    ps = rg.page_size
    tseq = rg.token_seq()
    seqs = sorted({int(tseq[t]) for t in tokens})
    # compact batch of the sampled requests: all their query tokens (positions
    # depend on q_len) and their page-table entries, renumbered
    q_lens = rg.q_lens[seqs]
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int64)
    npg = -(-rg.seq_lens[seqs].astype(np.int64) // ps)
    cu_kv = np.concatenate([[0], np.cumsum(npg * ps)]).astype(np.int64)
    ent = np.concatenate([int(rg.cu_kv_lens[s]) // ps + np.arange(n) for s, n in zip(seqs, npg)])
    phys = rg.page_indices[ent].astype(np.int64)
    pos_of = {s: i for i, s in enumerate(seqs)}
    ctok = [int(cu_q[pos_of[int(tseq[t])]] + t - int(rg.cu_q_lens[int(tseq[t])])) for t in tokens]
    meta = dict(seq_lens=rg.seq_lens[seqs].astype(np.int64), cu_q_lens=cu_q, cu_kv_lens=cu_kv)
    dev = wl.kcache[0].device
    tidx = torch.tensor(tokens, dtype=torch.long, device=wl.q_idx.device)
    q_idx = dict(zip(ctok, _host_bits(wl.q_idx.index_select(0, tidx))))
    w = dict(zip(ctok, _host_bits(wl.w.index_select(0, tidx.to(wl.w.device)))))
    pidx = torch.from_numpy(phys).to(dev)
    types = list(wl.indexer_types) if wl.indexer_types else [0]
    full_slot, src_slot, nfull = O.build_index_share_map(["full" if x == 0 else "shared" for x in types], 0,
                                                         len(types))
    kcaches = [_host_bits(wl.kcache[i].index_select(0, pidx)) for i in range(nfull)]
    pi_idx = np.arange(len(phys), dtype=np.int64)  # the compacted indexer pools are in page-table order
    seconds = 0.0
    sels = {}
    use_pages = prefill or page_budget is not None
    for slot in range(nfull):
        t0 = time.perf_counter()
        if use_pages:
            sel, rows = O.indexer_page_topk(q_idx, w, kcaches[slot], page_indices=pi_idx,
                                            k_pages=page_budget or wl.k_pages, tokens=ctok, **meta)
            if prefill:  # the prefill step also keeps the token top-k
                O.topk_rows_of(rows, wl.k)
        else:
            sel, rows = O.indexer_topk(q_idx, w, kcaches[slot], page_indices=pi_idx, k=wl.k, tokens=ctok,
                                       **meta)
        seconds += time.perf_counter() - t0
        sels[slot] = sel
    for layer in range(len(types)):
        sel = sels[src_slot[layer]]
        # attention pool: the physical pages the selections name, plus a zero page
        need = set()
        for i, t in enumerate(ctok):
            s = pos_of[int(tseq[tokens[i]])]
            row = sel[i][sel[i] >= 0].astype(np.int64)
            pages = row if use_pages else np.unique(row // ps)
            need.update((int(cu_kv[s]) // ps + pages).tolist())
        need = np.array(sorted(need), np.int64)
        apool = _host_bits(wl.kv[layer].index_select(0, torch.from_numpy(phys[need]).to(dev)))
        apool = np.concatenate([np.zeros((1,) + apool.shape[1:], apool.dtype), apool])
        api = np.zeros(len(phys), np.int64)
        api[need] = np.arange(1, len(need) + 1)
        qrows = dict(zip(ctok, _host_bits(wl.q[layer].index_select(0, tidx.to(wl.q[layer].device)))))
        selrows = dict(zip(ctok, sel))
        t0 = time.perf_counter()
        O.sparse_mla(qrows, apool, page_indices=api, sel=selrows, unit=ps if use_pages else 1,
                     sm_scale=wl.sm_scale, Dv=MLA_DV, tokens=ctok, **meta)
        seconds += time.perf_counter() - t0
    return seconds


def oracle_estimate(wl, tokens, prefill, page_budget=None):
    """The oracle's time for one full step of the workload, extrapolated from
    the sampled rows by counted work: the oracle's loops cost in proportion to
    its score pairs (2*32*128 FLOP each, per full layer) and attended keys
    (2*H*(576+512) FLOP each, per layer; counted as the selection size capped
    by the visible prefix), so the full step is estimated at the sample's
    seconds x full work / sample work."""
    import numpy as np

    secs = oracle_sample_seconds(wl, tokens, prefill, page_budget)
    types = list(wl.indexer_types) if wl.indexer_types else [0]
    nfull, nl = sum(1 for x in types if x == 0), len(types)
    nvis, att = row_work(wl, prefill, page_budget)
    flop_att = 2 * wl.H * (MLA_DK + MLA_DV)

    def work(idx):
        return nfull * IDX_FLOP_PER_PAIR * float(nvis[idx].sum()) + nl * flop_att * float(att[idx].sum())

    w_full = work(slice(None))
    w_smp = work(np.asarray(tokens, np.int64))
    return secs * w_full / max(w_smp, 1.0), secs, len(tokens)


def _workload_device():
    import torch

    return torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")


def cpu_baseline_line(wl, prefill, page_budget, name, target_s=15.0):
    """The oracle on the host cores on a bounded row sample of the workload,
    extrapolated to one full step by counted work, as tokens/s."""
    import oracle as O

    n = 64 if prefill else 48
    toks = sample_tokens(wl, n, seed=1)
    est, secs, nrow = oracle_estimate(wl, toks, prefill, page_budget)
    if secs < target_s / 3 and nrow < wl.rg.T:  # too small to time well: one larger sample
        scale = min(8.0, target_s / max(secs, 1e-3))
        toks = sample_tokens(wl, int(n * scale), seed=2)
        est, secs, nrow = oracle_estimate(wl, toks, prefill, page_budget)
    return {"value": wl.rg.T / est, "unit": "tokens/s", "cores": O.num_threads(), "kind": "oracle",
            "cpu": cpu_model(), "oracle_seconds": secs, "extrapolated_step_s": est,
            "sample": f"{nrow} of {wl.rg.T} query rows of {name} (stratified: decode rows and rows spread "
                      f"over every extend), every layer of the step on those rows; the step's time is "
                      f"extrapolated from the sample by counted work (score pairs and attended keys)"}


# --------------------------------------------------------------- reference
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import dsa_inputs as DI
    import oracle as O

    dev = _workload_device()
    wl = DI.WORKLOADS[args.workload](device=dev)
    rg = wl.rg
    prefill = bool((rg.q_lens > 1).any())
    rows_per_step = 16
    ests, secs, nrows = [], 0.0, 0
    for i in range(args.warmup + args.steps):
        toks = sample_tokens(wl, rows_per_step, seed=100 + i)
        est, s, n = oracle_estimate(wl, toks, prefill)
        if i >= args.warmup:
            ests.append(est)
            secs += s
            nrows += n
    total = sum(ests)
    value = rg.T * args.steps / total
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, "tokens_per_step": rg.T, "layers": len(wl.indexer_types or [0]),
                   "sample": f"{rows_per_step} query rows per step (stratified), extrapolated by counted work"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": O.num_threads(), "kind": "oracle",
                         "cpu": cpu_model(), "oracle_seconds": secs,
                         "sample": f"{nrows} query rows of {args.workload} over {args.steps} steps; each step's "
                                   f"time extrapolated from its rows by counted work"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- ours
def make_timer(flush):
    import torch

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

    return timed


def capture_step(rn, dev, warmup):
    """CUDA graph of one step (the launch overhead of the small kernels
    removed), or None if capture fails."""
    import torch

    try:
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                rn.step()
        torch.cuda.current_stream(dev).wait_stream(s)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        return g
    except Exception:  # pragma: no cover - reported in the JSON line
        torch.cuda.synchronize()
        return None


def time_steps(run, flush, steps):
    import torch

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record()
        run()
        ends[i].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def side_workload(name, dev, flush, args):
    """Step time and per-stage rooflines of another workload (one layer per
    step), for the headline line's ``workloads`` object."""
    import torch

    import dsa_inputs as DI
    from deepseek_sparse_attention_score_gb300.layer import LayerRunner

    wl = DI.WORKLOADS[name](device=dev)
    rn = LayerRunner(wl, dev)
    for _ in range(max(1, args.warmup)):
        rn.step()
    torch.cuda.synchronize()
    assert rn.status.item() == 0, f"{name}: device status {rn.status.item():#x}"
    g = capture_step(rn, dev, args.warmup)
    ms = time_steps(g.replay if g is not None else rn.step, flush, args.steps)
    timed = make_timer(flush)
    kern = stage_roofline(wl, rn, timed)
    step_ms = sum(ms) / len(ms)
    res = {"tokens_per_s": rn.T / (step_ms * 1e-3), "ms_per_step": step_ms, "tokens_per_step": rn.T,
           "kv_len": KV_LEN_DESC.get(name), "cuda_graph": g is not None, "kernels": kern}
    dom = dominant_stage(kern)
    res["dominant"] = {"kernel": dom, "frac": kern[dom]["frac"], "bound": kern[dom]["bound"],
                       "traffic": committed_traffic(dom, name)}
    del rn, wl, g
    torch.cuda.empty_cache()
    return res


def run_ours(args):
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

    graph = capture_step(rn, dev, args.warmup)
    run = graph.replay if graph is not None else rn.step

    with ClockSampler(torch.cuda.current_device()) as clk:
        # keep the GPU busy with back-to-back steps for ~1.5 s around the timed
        # steps so the 200 ms clock samples land under the same load
        t_end = time.perf_counter() + 1.0
        while time.perf_counter() < t_end:
            for _ in range(4):
                flush.zero_()
                run()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        step_ms = time_steps(run, flush, args.steps)
        wall = time.perf_counter() - w0
        barrier()
        t_end = time.perf_counter() + 0.5
        while time.perf_counter() < t_end:
            for _ in range(4):
                flush.zero_()
                run()
            torch.cuda.synchronize()
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    value = replica_throughput(T, args.steps, world, total_s)
    clocks = clk.summary()

    # per-ABI-call times (eager, L2 flushed before each) for the roofline
    timed = make_timer(flush)
    kern = stage_roofline(wl, rn, timed)
    dom = dominant_stage(kern)
    d = kern[dom]
    roof = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"], "unit": d["unit"],
            "frac": d["frac"], "peak_kind": d["peak_kind"], "traffic": committed_traffic(dom, args.workload)}

    # end to end through the public API with host buffers
    pin = lambda t: t.detach().to("cpu").pin_memory()
    h_q_idx, h_w = pin(rn.q_idx), pin(rn.w)
    h_q = [pin(x) for x in rn.q]
    h_meta = [pin(m) for m in rn.meta]
    h_new_kv = [pin(x) for x in rn.new_kv]
    h_new_k = [pin(x) for x in rn.new_k]
    h_topk = torch.empty(rn.topk[0].shape, dtype=torch.int32).pin_memory()
    h_o = [torch.empty(x.shape, dtype=torch.bfloat16).pin_memory() for x in rn.o]
    h2d = sum(t.numel() * t.element_size() for t in [h_q_idx, h_w, *h_q, *h_meta, *h_new_kv, *h_new_k])
    d2h = h_topk.numel() * 4 + sum(x.numel() * 2 for x in h_o)

    # the whole host-buffer step (copies on two streams, kernels) as one
    # CUDA graph; every replay copies the inputs in and the outputs out
    side = torch.cuda.Stream(dev)
    e2e_eager = lambda: rn.step_host(h_q_idx, h_w, h_q, h_meta, h_topk, h_o, side, h_new_kv, h_new_k)
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
    e_ms = make_timer(flush)
    e_list = [e_ms(e2e_step, reps=1) for _ in range(args.steps)]
    e2e_s = max_over_ranks(sum(e_list) / 1e3, world)
    e2e = {"value": replica_throughput(T, args.steps, world, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * e2e_s / args.steps, "cuda_graph": e2e_graph}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_line(wl, rn.prefill, rn.page_budget, args.workload)

    config = {"workload": args.workload, "requests": wl.rg.S, "tokens_per_step": T, "layers": len(rn.types),
              "kv_len": KV_LEN_DESC.get(args.workload, "per request, from the workload"),
              "k": wl.k, "k_pages": wl.k_pages, "mla_heads": wl.H, "page_size": wl.rg.page_size,
              "l2": "flushed (512 MB write) before every timed step", "cuda_graph": graph is not None,
              "parallelism": "replicas" if world > 1 else "single"}
    # free the headline workload before the side workloads are built
    del rn, wl, graph, h_q, h_o, h_q_idx, h_w, h_meta, h_topk, h_new_kv, h_new_k
    torch.cuda.empty_cache()
    sides = {}
    if not args.only and rank == 0 and world == 1:
        for name in SIDE_WORKLOADS:
            if name != args.workload:
                sides[name] = side_workload(name, dev, flush, args)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
            "roofline": roof, "kernels": kern, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
            "clocks": clocks, "clock_window": "1.5 s of back-to-back steps enclosing the timed steps",
            "wall_s_timed_region": wall, "workloads": sides,
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

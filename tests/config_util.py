"""Helpers for the full-size workload parity tests: host copies of only the
rows and pages a sample of query tokens touches, so the CPU oracle can check
them one by one."""
from __future__ import annotations

import numpy as np
import torch


def rows_of(t: torch.Tensor, tokens):
    """{token: fp32 numpy row} for a device tensor indexed by token."""
    idx = torch.as_tensor(sorted(set(int(x) for x in tokens)), dtype=torch.long, device=t.device)
    vals = t.index_select(0, idx).float().cpu().numpy()
    return {int(k): v for k, v in zip(idx.tolist(), vals)}


class CompactPool:
    """A compacted copy of the physical pages a check needs, plus the page
    table remapped onto it (entries whose page was not copied point at a
    zero page, and are never read by the checks that use the pool)."""

    def __init__(self, caches, page_indices, entries):
        pi = np.asarray(page_indices, dtype=np.int64)
        entries = np.unique(np.asarray(list(entries), dtype=np.int64))
        phys = np.unique(pi[entries])
        self.remap = np.zeros(int(max(pi.max(), 0)) + 1, dtype=np.int64)
        self.remap[phys] = np.arange(1, len(phys) + 1)
        self.page_indices = self.remap[pi].astype(np.int32)
        idx = torch.as_tensor(phys, dtype=torch.long, device=caches[0].device)
        self.caches = []
        for c in caches:
            sub = c.index_select(0, idx).float().cpu().numpy()
            z = np.zeros((1,) + sub.shape[1:], dtype=np.float32)
            self.caches.append(np.concatenate([z, sub], axis=0))


def seq_entries(rg, seqs):
    """Page-table entries of whole requests."""
    out = []
    for s in seqs:
        b = int(rg.cu_kv_lens[s]) // rg.page_size
        out.extend(range(b, b + -(-int(rg.seq_lens[s]) // rg.page_size)))
    return out


def sel_entries(rg, token_seq, tokens, sel, unit):
    """Page-table entries named by the selections of the given tokens."""
    ps = rg.page_size
    out = []
    for t in tokens:
        s = int(token_seq[t])
        b = int(rg.cu_kv_lens[s]) // ps
        row = np.asarray(sel[t])
        row = row[row >= 0]
        pages = np.unique(row // ps) if unit == 1 else np.unique(row)
        out.extend((b + pages).tolist())
    return out

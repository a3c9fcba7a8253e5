"""Helpers shared by the GPU parity tests: moving seeded workloads to the
device, and the comparison rules of the parity bar."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

TOPK_REL_BAND = 1e-3     # top-k near-tie band, relative to the k-th score
SCORE_RTOL = 1e-3        # indexer score tolerance (relative)
ATTN_REL_L2 = 1e-2       # attention output, relative L2
ATTN_MAX_ABS = 3e-2      # attention output, max abs


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def meta_to(rg, dev):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in
            (rg.seq_lens, rg.cu_q_lens, rg.cu_kv_lens, rg.page_indices)]


def meta_np(rg):
    return dict(seq_lens=rg.seq_lens, cu_q_lens=rg.cu_q_lens, cu_kv_lens=rg.cu_kv_lens,
                page_indices=rg.page_indices)


def check_topk_rows(got, ref_rows, k, scores_rows, what="top-k"):
    """Selected sets must be equal except positions whose oracle score lies
    within TOPK_REL_BAND (relative) of the k-th score; the rest of the
    row must still be valid (unique, visible, the right count)."""
    got = np.asarray(got)
    bad = []
    for r, (g, ref, s) in enumerate(zip(got, ref_rows, scores_rows)):
        n = len(s)
        gs = g[g >= 0]
        assert len(gs) == min(k, n), (what, r, len(gs), min(k, n))
        assert len(np.unique(gs)) == len(gs), (what, r, "duplicates")
        assert np.all(np.diff(gs) > 0), (what, r, "not ascending")
        assert np.all(gs < n), (what, r, "invisible position selected")
        assert np.all(g[len(gs):] == -1), (what, r, "padding")
        rs = ref[ref >= 0]
        if n <= k:
            assert np.array_equal(gs, np.arange(n)), (what, r)
            continue
        kth = np.sort(s.astype(np.float64))[::-1][k - 1]
        band = np.abs(s.astype(np.float64) - kth) <= TOPK_REL_BAND * max(abs(kth), 1e-30)
        a = set(gs.tolist()) - set(np.nonzero(band)[0].tolist())
        b = set(rs.tolist()) - set(np.nonzero(band)[0].tolist())
        if a != b:
            bad.append((r, sorted(a ^ b)[:8]))
    assert not bad, f"{what}: {len(bad)} rows differ outside the near-tie band, e.g. {bad[:3]}"


def check_scores(got_vals, got_idx, scores_rows):
    for g, i, s in zip(np.asarray(got_vals), np.asarray(got_idx), scores_rows):
        m = i >= 0
        ref = s[i[m]].astype(np.float64)
        v = g[m].astype(np.float64)
        denom = np.maximum(np.abs(ref), 1e-6 * max(np.abs(s).max(), 1e-30))
        assert np.all(np.abs(v - ref) <= SCORE_RTOL * denom), np.max(np.abs(v - ref) / denom)
        assert np.all(np.isneginf(g[~m]))


def check_attention(o_gpu, o_ref, what="attention"):
    o = f32(o_gpu).astype(np.float64) if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu, np.float64)
    err = o - o_ref
    nrm = np.linalg.norm(o_ref)
    rel = np.linalg.norm(err) / nrm if nrm > 0 else np.linalg.norm(err)
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= ATTN_REL_L2 and mx <= ATTN_MAX_ABS, f"{what}: rel-L2 {rel:.3e}, max-abs {mx:.3e}"
    return rel, mx


def member_bits_to_int8(member_words, QB):
    """[nQB, u_max, QB/32] uint32 words -> [nQB, QB, u_max] int8 (the pages'
    membership layout)."""
    w = np.asarray(member_words).astype(np.uint32)
    nqb, u_max, nw = w.shape
    bits = ((w[:, :, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(nqb, u_max, nw * 32)
    return bits.transpose(0, 2, 1).astype(np.int8)[:, :QB, :]

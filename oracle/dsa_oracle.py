"""CPU oracle for the DSA sparse-attention hot path (test infrastructure only).

This is the plain, slow, obviously correct definition of every step of the
path, written from the sglang-jax DSA pages:

  * "ref.py" (jnp reference implementations): ``build_index_share_map``,
    ``streamindex_topk_ref``, ``streamindex_page_topk_ref``, ``sparse_mla_ref``;
  * "sparse_mla_prefill_qblock.py" (blocked sparse-MLA prefill):
    ``build_block_unit_tables``, ``_qblock_kernel``,
    ``sparse_mla_attention_qblock``, ``prefill_write_and_attend_ragged_qblock``;
  * "dsa_sparse_backend.py" (DSA sparse attention backend): the IndexShare
    dispatch, the page budget of the prefill page top-k, and the paged cache
    write of the new tokens (``_scatter_paged``) that precedes the path.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module. It shares no code with the CUDA library and
imports nothing from it. Floating point is fp64 (bf16 inputs are widened
exactly); the indexer score is rounded once to fp32, as the pages keep scores
in fp32. The approximate top-k of the pages (``approx_max_k``) is replaced by
the exact top-k, ties going to the lower index.

Readings taken where the pages are silent:
  * selected sets are emitted in ascending index order, -1 padded (the pages
    emit score order; every consumer is order-invariant);
  * the attention masks every key by both ``j < kv_len`` and ``j <= pos``
    (the jnp reference applies only the first, the qblock kernel both; they
    coincide on indices produced by the indexer);
  * a row with no valid key outputs 0 (the pages' masked softmax does the same).

Queries may be given as arrays or as any mapping token -> row (so large
batches can be checked on a sample of rows); caches are arrays.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
and properties fixed outside this file (hand-worked examples, brute force on
tiny inputs, closed forms, reductions to library routines); none is
"parity unpinned".
"""
from __future__ import annotations

import numpy as np

NEG_INF = float("-inf")


# ---------------------------------------------------------------------------
# input widening and ragged metadata
# ---------------------------------------------------------------------------

def widen(x) -> np.ndarray:
    """Exact fp64 view of a tensor given as bf16 bit patterns (uint16/int16)
    or as an fp32/fp64 array."""
    x = np.asarray(x)
    if x.dtype in (np.uint16, np.int16):
        return (x.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def token_seq(cu_q_lens, T=None) -> np.ndarray:
    """Request of each query token: the ``s`` with
    ``cu_q_lens[s] <= t < cu_q_lens[s+1]`` (the searchsorted over
    ``cu_q_lens[1:]`` with side="right" of prefill_write_and_attend_ragged_qblock)."""
    cu = np.asarray(cu_q_lens, dtype=np.int64)
    if T is None:
        T = int(cu[-1])
    t = np.arange(T, dtype=np.int64)
    return np.searchsorted(cu[1:], t, side="right").astype(np.int64)


def token_pos(seq_lens, cu_q_lens) -> np.ndarray:
    """Absolute position of each query token,
    ``abs_q = kv_len - (q_end - q_start) + (t - q_start)`` (ref.py,
    streamindex_topk_ref, general path)."""
    sl = np.asarray(seq_lens, dtype=np.int64)
    cu = np.asarray(cu_q_lens, dtype=np.int64)
    s = token_seq(cu)
    t = np.arange(int(cu[-1]), dtype=np.int64)
    return sl[s] - (cu[s + 1] - cu[s]) + (t - cu[s])


def visible_len(seq_lens, cu_q_lens) -> np.ndarray:
    """Number of key positions token t may see: ``j < kv_len`` and ``j <= abs_q``
    (the mask of streamindex_topk_ref). The visible set is always the prefix
    ``[0, n)`` with ``n = clip(min(kv_len, abs_q + 1), 0)``."""
    sl = np.asarray(seq_lens, dtype=np.int64)
    s = token_seq(cu_q_lens)
    pos = token_pos(seq_lens, cu_q_lens)
    return np.clip(np.minimum(sl[s], pos + 1), 0, None)


def physical_rows(cu_kv_lens, page_indices, ps, s, positions) -> np.ndarray:
    """Flat row ``page*ps + offset`` of sequence-local key positions: request
    ``s`` owns the packed page-table entries starting at ``cu_kv_lens[s]//ps``
    (ref.py, ``seq_pages = page_indices[cu_kv_lens[s]//ps : ...]``)."""
    positions = np.asarray(positions, dtype=np.int64)
    base = int(cu_kv_lens[s]) // ps
    pages = np.asarray(page_indices, dtype=np.int64)[base + positions // ps]
    return pages * ps + positions % ps


# ---------------------------------------------------------------------------
# a7: IndexShare layer -> slot map
# ---------------------------------------------------------------------------

class ShareMapError(ValueError):
    pass


def build_index_share_map(indexer_types, skip_offset, num_layers):
    """ref.py, ``build_index_share_map``: a "full" layer opens a new slot, a
    "shared" layer consumes the nearest preceding full layer's slot; a shared
    layer with no preceding full layer, or an unknown type, is an error.
    ``None`` means every layer is full. ``skip_offset`` is accepted and, as on
    the page, not used."""
    del skip_offset
    if indexer_types is None:
        indexer_types = ["full"] * num_layers
    if len(indexer_types) != num_layers:
        raise ShareMapError("indexer_types length != num_layers")
    full_slot, src_slot = {}, {}
    last = -1
    for layer, kind in enumerate(indexer_types):
        if kind == "full":
            last = len(full_slot)
            full_slot[layer] = last
            src_slot[layer] = last
        elif kind == "shared":
            if last < 0:
                raise ShareMapError(f"layer {layer} is shared but no preceding full layer")
            src_slot[layer] = last
        else:
            raise ShareMapError(f"unknown indexer type {kind!r} at layer {layer}")
    return full_slot, src_slot, len(full_slot)


# ---------------------------------------------------------------------------
# a1: lightning-indexer score
# ---------------------------------------------------------------------------

def indexer_score_row(q_t, w_t, keys) -> np.ndarray:
    """Score of one query token against the rows of ``keys`` ([n, D]):
    ``s_j = sum_h relu(q[h,:] . k_j) * w[h]`` (ref.py, streamindex_topk_ref:
    an einsum over D, relu, an einsum with the head weights). Accumulated in
    fp64 and rounded once to fp32. No extra scale factor: the pages' score has
    none."""
    q_t = widen(q_t)  # [H, D]
    w_t = widen(w_t)  # [H]
    keys = widen(keys)  # [n, D]
    dots = q_t @ keys.T  # [H, n]
    s = (np.maximum(dots, 0.0) * w_t[:, None]).sum(axis=0)
    return s.astype(np.float32)


def indexer_scores(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens=None):
    """Score rows for the given tokens (all by default). Row ``t`` holds the
    scores of the visible prefix ``[0, visible_len[t])``; every other position
    is masked (-inf) and so is simply absent from the row."""
    kc = np.asarray(kcache)
    P, ps, D = kc.shape
    flat = kc.reshape(P * ps, D)
    seq = token_seq(cu_q_lens)
    nvis = visible_len(seq_lens, cu_q_lens)
    if tokens is None:
        tokens = range(len(seq))
    rows = []
    for t in tokens:
        n = int(nvis[t])
        r = physical_rows(cu_kv_lens, page_indices, ps, int(seq[t]), np.arange(n))
        rows.append(indexer_score_row(q[t], w[t], flat[r]) if n else np.zeros(0, np.float32))
    return rows


# ---------------------------------------------------------------------------
# a2 / a3: exact top-k over tokens and over max-pooled pages
# ---------------------------------------------------------------------------

def topk_of_row(scores, k) -> np.ndarray:
    """Exact top-k of one row: order the finite entries by (score desc, index
    asc), keep ``min(k, n)`` of them, emit them in ascending index order, pad
    with -1 (streamindex_topk_ref with exact selection; masked entries are
    never selected)."""
    scores = np.asarray(scores, dtype=np.float32)
    idx = np.nonzero(np.isfinite(scores))[0]
    order = np.lexsort((idx, -scores[idx].astype(np.float64)))
    chosen = np.sort(idx[order[: min(k, len(idx))]])
    out = np.full(k, -1, dtype=np.int32)
    out[: len(chosen)] = chosen
    return out


def page_scores_of_row(scores, ps) -> np.ndarray:
    """Max-pool a token score row per page of ``ps`` positions
    (streamindex_page_topk_ref: ``scores.reshape(.., pages, ps).max(-1)``);
    only visible positions enter the max, so every page of the visible prefix
    has a finite score."""
    scores = np.asarray(scores, dtype=np.float32)
    n = len(scores)
    npg = (n + ps - 1) // ps
    pad = np.full(npg * ps, -np.inf, dtype=np.float32)
    pad[:n] = scores
    return pad.reshape(npg, ps).max(axis=1)


def page_topk_of_row(scores, ps, k_pages) -> np.ndarray:
    """streamindex_page_topk_ref: top ``k_pages`` pages by max-pooled score,
    pages with score -inf dropped, sequence-local page ids (exact, ties to the
    lower page, ascending output, -1 padded)."""
    return topk_of_row(page_scores_of_row(scores, ps), k_pages)


def indexer_topk(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, k, tokens=None):
    rows = indexer_scores(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens)
    return np.stack([topk_of_row(r, k) for r in rows]) if rows else np.zeros((0, k), np.int32), rows


def indexer_page_topk(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, k_pages,
                      tokens=None):
    kc = np.asarray(kcache)
    ps = kc.shape[1]
    rows = indexer_scores(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens)
    out = [page_topk_of_row(r, ps, k_pages) for r in rows]
    return (np.stack(out) if out else np.zeros((0, k_pages), np.int32)), rows


# ---------------------------------------------------------------------------
# a4: per-query-block union and membership
# ---------------------------------------------------------------------------

def lift_units(topk_units, cu_q_lens, cu_kv_lens, ps) -> np.ndarray:
    """Lift sequence-local page ids to global page-table keys,
    ``g = cu_kv_lens[seq(t)]//ps + p`` for ``p >= 0``, else -1
    (sparse_mla_attention_qblock, ragged mode)."""
    tk = np.asarray(topk_units, dtype=np.int64)
    seq = token_seq(cu_q_lens, tk.shape[0])
    base = np.asarray(cu_kv_lens, dtype=np.int64)[seq] // ps
    return np.where(tk >= 0, tk + base[:, None], -1)


def block_union(units_global, QB, u_max):
    """build_block_unit_tables: pad T to a multiple of QB with -1 rows; per
    block the ascending unique list of the selected ids (kept up to
    ``u_max``, -1 padded), the true (uncapped) union size, and the membership
    ``member[b, q, u] = 1`` iff query q of block b selected ``units[b, u]``."""
    g = np.asarray(units_global, dtype=np.int64)
    T, K = g.shape
    nqb = -(-T // QB) if T else 0
    units = np.full((nqb, u_max), -1, dtype=np.int32)
    member = np.zeros((nqb, QB, u_max), dtype=np.int8)
    counts = np.zeros(nqb, dtype=np.int32)
    for b in range(nqb):
        blk = g[b * QB: min(T, (b + 1) * QB)]
        uniq = np.unique(blk[blk >= 0])
        counts[b] = len(uniq)
        kept = uniq[:u_max]
        units[b, : len(kept)] = kept
        for q in range(blk.shape[0]):
            sel = blk[q][blk[q] >= 0]
            member[b, q, : len(kept)] = np.isin(kept, sel)
    return units, member, counts


# ---------------------------------------------------------------------------
# a5 / a6: absorbed-MLA sparse attention
# ---------------------------------------------------------------------------

def _masked_softmax_attend(q_t, keys, vals, sm_scale):
    """fp64 masked-softmax attention of one token over the given (already
    filtered) keys. Returns (o [H, Dv], lse [H]); no key gives o = 0 and
    lse = -inf (sparse_mla_ref: ``p = where(valid, softmax, 0)``)."""
    H = q_t.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((H, vals.shape[1])), np.full(H, NEG_INF)
    logits = sm_scale * (q_t @ keys.T)  # [H, n]
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    l = e.sum(axis=1, keepdims=True)
    o = (e @ vals) / l
    return o, (m + np.log(l))[:, 0]


def selected_positions(sel_row, unit, ps):
    """Key positions named by one selection row: token ids (``unit == 1``) or
    whole pages expanded to ``p*ps .. p*ps+ps-1`` (``unit == ps``). -1 entries
    are ignored; duplicates are kept as given."""
    sel = np.asarray(sel_row, dtype=np.int64)
    sel = sel[sel >= 0]
    if unit == 1:
        return sel
    return (sel[:, None] * unit + np.arange(unit)[None, :]).reshape(-1)


def sparse_mla(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, sel, unit, sm_scale, Dv,
               tokens=None):
    """sparse_mla_ref: for each token, masked softmax of
    ``sm_scale * q[t,h,:] . kv[j,:Dk]`` over the selected positions j with
    ``0 <= j < kv_len`` and ``j <= pos(t)``, output ``sum_j p_j kv[j, :Dv]``.
    Returns fp64 ``o [n, H, Dv]`` and ``lse [n, H]``."""
    kvc = np.asarray(kv)
    P, ps, Dk_row = kvc.shape
    flat = kvc.reshape(P * ps, Dk_row)
    seq = token_seq(cu_q_lens)
    nvis = visible_len(seq_lens, cu_q_lens)
    if tokens is None:
        tokens = range(len(seq))
    os_, ls = [], []
    for t in tokens:
        j = selected_positions(sel[t], unit, ps)
        j = j[(j >= 0) & (j < nvis[t])]
        rows = widen(flat[physical_rows(cu_kv_lens, page_indices, ps, int(seq[t]), j)])
        qt = widen(q[t])
        Dk = qt.shape[-1]
        o, l = _masked_softmax_attend(qt, rows[:, :Dk], rows[:, :Dv], sm_scale)
        os_.append(o)
        ls.append(l)
    return np.stack(os_), np.stack(ls)


def qblock_attend(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, units, member, counts,
                  QB, sm_scale, Dv, tokens=None):
    """_qblock_kernel semantics: query t of block b walks the block's union
    slots ``u < min(count, u_max)`` in order; unit ``g = units[b,u]`` covers
    physical page ``page_indices[g]`` whose row r is key position
    ``kp = g*ps + r - base_tok(t)``; the key is visible iff
    ``member[b,q,u]`` and ``kp <= pos(t)`` and ``kp < kv_len(t)``. Masked
    softmax over the visible keys; a row with none outputs 0."""
    kvc = np.asarray(kv)
    P, ps, Dk_row = kvc.shape
    flat = kvc.reshape(P * ps, Dk_row)
    seq = token_seq(cu_q_lens)
    pos = token_pos(seq_lens, cu_q_lens)
    sl = np.asarray(seq_lens, dtype=np.int64)
    pi = np.asarray(page_indices, dtype=np.int64)
    u_max = units.shape[1]
    if tokens is None:
        tokens = range(len(seq))
    os_, ls = [], []
    for t in tokens:
        b, qq = divmod(int(t), QB)
        s = int(seq[t])
        base_tok = (int(cu_kv_lens[s]) // ps) * ps
        rows_sel = []
        for u in range(min(int(counts[b]), u_max)):
            if not member[b, qq, u]:
                continue
            g = int(units[b, u])
            kp = g * ps + np.arange(ps) - base_tok
            ok = (kp <= pos[t]) & (kp < sl[s])
            rows_sel.append((pi[g] * ps + np.arange(ps))[ok])
        r = np.concatenate(rows_sel) if rows_sel else np.zeros(0, np.int64)
        rows = widen(flat[r])
        qt = widen(q[t])
        Dk = qt.shape[-1]
        o, l = _masked_softmax_attend(qt, rows[:, :Dk], rows[:, :Dv], sm_scale)
        os_.append(o)
        ls.append(l)
    return np.stack(os_), np.stack(ls)


def dense_mla(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, sm_scale, Dv, tokens=None,
              sliding_window=None, soft_cap=None):
    """Dense causal absorbed-MLA (the route the backend falls back to): every
    visible position ``j < min(kv_len, pos+1)``, one position at a time, with
    a two-pass max/sum softmax. Written independently of ``sparse_mla`` so the
    property "top-k with k >= kv_len equals dense attention" pins both.

    The backend's dense route (dsa_sparse_backend.py, ``_run_dense``) also
    passes the layer's ``sliding_window`` and ``logit_cap`` to the dense
    kernel, whose module the pages do not show; the plain readings taken:
    a window W keeps the W most recent positions ``pos - W < j <= pos``, and a
    cap c maps each scaled logit l to ``c * tanh(l / c)`` before the softmax."""
    kvc = np.asarray(kv)
    P, ps, Dk_row = kvc.shape
    seq = token_seq(cu_q_lens)
    nvis = visible_len(seq_lens, cu_q_lens)
    pi = np.asarray(page_indices, dtype=np.int64)
    if tokens is None:
        tokens = range(len(seq))
    out = []
    for t in tokens:
        s = int(seq[t])
        qt = widen(q[t])
        H = qt.shape[0]
        Dk = qt.shape[-1]
        n = int(nvis[t])
        lo = 0
        if sliding_window:
            pos = n - 1  # the last visible position is the query's own
            lo = max(0, pos - int(sliding_window) + 1)
        if n - lo <= 0:
            out.append(np.zeros((H, Dv)))
            continue
        base = int(cu_kv_lens[s]) // ps
        logit = np.empty((n - lo, H))
        vals = np.empty((n - lo, Dv))
        for j in range(lo, n):
            row = widen(kvc[pi[base + j // ps], j % ps])
            l = sm_scale * (qt @ row[:Dk])
            logit[j - lo] = soft_cap * np.tanh(l / soft_cap) if soft_cap else l
            vals[j - lo] = row[:Dv]
        mx = logit.max(axis=0)
        wgt = np.exp(logit - mx)
        out.append((wgt.T @ vals) / wgt.sum(axis=0)[:, None])
    return np.stack(out)


# ---------------------------------------------------------------------------
# the step before the path: paged write-back of the new tokens' rows
# ---------------------------------------------------------------------------

def paged_write_back(cache, rows, seq_lens, cu_q_lens, cu_kv_lens, page_indices):
    """Copy of ``cache`` [P, ps, W] with every query token's row written at its
    own slot (dsa_sparse_backend.py, ``_scatter_paged``): token t of request s
    lands at absolute position ``pos = kv_len - q_len + (t - q_start)``, i.e.
    row ``pos % ps`` of physical page ``page_indices[cu_kv_lens[s]//ps +
    pos//ps]``; the first ``rows.shape[1]`` columns are overwritten. The
    pages' padding rows (sent to a sentinel page) do not occur here: every
    token belongs to a request."""
    out = np.array(cache, copy=True)
    ps = out.shape[1]
    D = np.asarray(rows).shape[1]
    cu = np.asarray(cu_q_lens, dtype=np.int64)
    seq = token_seq(cu)
    pos = token_pos(seq_lens, cu)
    for t in range(int(cu[-1])):
        s = int(seq[t])
        entry = int(cu_kv_lens[s]) // ps + int(pos[t]) // ps
        out[int(page_indices[entry]), int(pos[t]) % ps, :D] = rows[t][:D]
    return out


def topk_pages_of_tokens(topk_row, ps, cap):
    """Page list of one query's token selections (dsa_sparse_backend.py,
    ``compute_topk_pages``, whose module the pages import but do not show;
    the plain reading): the ascending unique pages ``position // ps`` of the
    selected tokens, the first ``cap`` of them, -1 padded; also the uncapped
    number of unique pages."""
    row = np.asarray(topk_row, dtype=np.int64)
    uniq = np.unique(row[row >= 0] // ps)
    out = np.full(cap, -1, dtype=np.int64)
    n = min(cap, len(uniq))
    out[:n] = uniq[:n]
    return out, len(uniq)


def approx_topk_of_row(scores, k, over):
    """Approximate top-k of one score row (the pages' fast path uses
    ``approx_max_k`` with a recall target; this is the two-stage form the
    build implements, written out): fold the n scores into
    ``B = min(n, over*k)`` bins (bin b holds positions b, b+B, ...), keep each
    bin's largest score (lowest position on ties), take the exact top-k of
    the B bin maxima (ties to the lower bin) and return their positions in
    ascending order, -1 padded."""
    s = np.asarray(scores, dtype=np.float32)
    n = len(s)
    out = np.full(k, -1, dtype=np.int64)
    if n == 0:
        return out
    B = min(n, over * k)
    best_pos = np.empty(B, dtype=np.int64)
    best_val = np.empty(B, dtype=np.float32)
    for b in range(B):
        idx = np.arange(b, n, B)
        j = idx[int(np.argmax(s[idx]))]  # argmax returns the first (lowest) maximum
        best_pos[b], best_val[b] = j, s[j]
    bins = topk_of_row(best_val, k)
    sel = np.sort(best_pos[bins[bins >= 0]])
    out[: len(sel)] = sel
    return out

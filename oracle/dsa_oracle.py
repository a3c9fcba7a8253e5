"""Python binding of the C++ CPU oracle (``oracle/dsa_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this module. It shares
no code with the CUDA library and imports nothing from it.

Every step of the method is computed in ``dsa_oracle.cpp`` (plain C++17, fp64,
OpenMP over query rows; see its header for the pages it follows and the
readings it takes). This module only marshals arguments: it picks the rows of
the requested tokens, passes arrays in their own element type (fp32, fp64 or
bf16 bit patterns, all widened exactly by the C++ side) and shapes the
results. Queries, weights and selections may be given as arrays indexed by
token or as any mapping token -> row, so large batches can be checked on a
sample of rows; caches are arrays.

The shared library is compiled from source on first use (``g++ -fopenmp``),
by ``build_oracle.build()``.
"""
from __future__ import annotations

import ctypes
from collections.abc import Mapping

import numpy as np

from . import build_oracle

NEG_INF = float("-inf")

_F32, _F64, _BF16 = 0, 1, 2
_P = ctypes.c_void_p
_L = ctypes.c_longlong
_D = ctypes.c_double
_lib = None


def _load():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build_oracle.build())
        sig = {
            "orc_num_threads": ([], ctypes.c_int),
            "orc_widen": ([_P, ctypes.c_int, _L, _P], None),
            "orc_token_seq": ([_P, _L, _L, _P], None),
            "orc_token_geometry": ([_P, _P, _L, _L, _P, _P, _P], None),
            "orc_physical_rows": ([_P, _P, _L, _L, _P, _L, _P], None),
            "orc_share_map": ([_P, _L, _L, _P, _P, _P], ctypes.c_int),
            "orc_score_row": ([_P, ctypes.c_int, _P, ctypes.c_int, _P, ctypes.c_int, _L, _L, _L, _P], None),
            "orc_indexer_scores": ([_P, ctypes.c_int, _P, ctypes.c_int, _P, ctypes.c_int, _L, _L, _L, _P, _P, _P,
                                    _P, _L, _P, _L, _L, _P, _P], None),
            "orc_topk_rows": ([_P, _L, _P, _L, _L, _P], None),
            "orc_page_topk_rows": ([_P, _L, _P, _L, _L, _L, _P], None),
            "orc_page_scores_row": ([_P, _L, _L, _P], None),
            "orc_lift_units": ([_P, _L, _L, _P, _L, _P, _L, _P], None),
            "orc_block_union": ([_P, _L, _L, _L, _L, _P, _P, _P], None),
            "orc_selected_positions": ([_P, _L, _L, _P], _L),
            "orc_sparse_mla": ([_P, ctypes.c_int, _P, ctypes.c_int, _L, _L, _L, _L, _L, _P, _P, _P, _P, _L, _P, _L,
                                _P, _L, _L, _D, _P, _P], None),
            "orc_qblock_attend": ([_P, ctypes.c_int, _P, ctypes.c_int, _L, _L, _L, _L, _L, _P, _P, _P, _P, _L, _P,
                                   _L, _P, _P, _P, _L, _L, _D, _P, _P], None),
            "orc_dense_mla": ([_P, ctypes.c_int, _P, ctypes.c_int, _L, _L, _L, _L, _L, _P, _P, _P, _P, _L, _P, _L,
                               _D, _L, _D, _P], None),
            "orc_paged_write_back": ([_P, _L, _L, _L, _P, _L, _P, _P, _P, _P, _L, _L], None),
            "orc_topk_pages_of_tokens": ([_P, _L, _L, _L, _P], _L),
            "orc_approx_topk_row": ([_P, _L, _L, _L, _P], None),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def num_threads() -> int:
    """Host threads the oracle's row loops run on (OpenMP)."""
    return int(_load().orc_num_threads())


# ---------------------------------------------------------------- marshalling
def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _typed(x):
    """(contiguous array, element-type code) with no rounding: fp32 and fp64
    pass as they are, int16/uint16 are bf16 bit patterns, anything else is
    converted to fp64."""
    a = np.asarray(x)
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), _F32
    if a.dtype == np.float64:
        return np.ascontiguousarray(a), _F64
    if a.dtype in (np.uint16, np.int16):
        return np.ascontiguousarray(a.view(np.uint16)), _BF16
    return np.ascontiguousarray(a.astype(np.float64)), _F64


def _rows(x, tokens):
    """The rows of ``tokens`` from an array indexed by token or a mapping."""
    if isinstance(x, Mapping):
        return np.stack([np.asarray(x[int(t)]) for t in tokens])
    a = np.asarray(x)
    if len(tokens) == a.shape[0] and np.array_equal(tokens, np.arange(a.shape[0])):
        return a
    return a[np.asarray(tokens, dtype=np.int64)]


def _meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices):
    return _i64(seq_lens), _i64(cu_q_lens), _i64(cu_kv_lens), _i64(page_indices)


def _tokens(tokens, cu_q_lens):
    if tokens is None:
        return np.arange(int(np.asarray(cu_q_lens)[-1]), dtype=np.int64)
    return _i64(list(tokens))


# ---------------------------------------------------- widening and metadata
def widen(x) -> np.ndarray:
    """Exact fp64 values of a tensor given as bf16 bit patterns (uint16/int16)
    or as an fp32/fp64 array."""
    a, dt = _typed(x)
    out = np.empty(a.shape, np.float64)
    _load().orc_widen(_p(a), dt, a.size, _p(out))
    return out


def _geometry(seq_lens, cu_q_lens):
    sl, cu = _i64(seq_lens), _i64(cu_q_lens)
    T = int(cu[-1])
    seq, pos, nvis = (np.empty(T, np.int64) for _ in range(3))
    _load().orc_token_geometry(_p(sl), _p(cu), len(cu) - 1, T, _p(seq), _p(pos), _p(nvis))
    return seq, pos, nvis


def token_seq(cu_q_lens, T=None) -> np.ndarray:
    """Request of each query token: the ``s`` with
    ``cu_q_lens[s] <= t < cu_q_lens[s+1]``."""
    cu = _i64(cu_q_lens)
    T = int(cu[-1]) if T is None else int(T)
    seq = np.empty(T, np.int64)
    _load().orc_token_seq(_p(cu), len(cu) - 1, T, _p(seq))
    return seq


def token_pos(seq_lens, cu_q_lens) -> np.ndarray:
    """Absolute position of each query token."""
    return _geometry(seq_lens, cu_q_lens)[1]


def visible_len(seq_lens, cu_q_lens) -> np.ndarray:
    """Visible prefix length of each token (``j < kv_len`` and ``j <= pos``)."""
    return _geometry(seq_lens, cu_q_lens)[2]


def physical_rows(cu_kv_lens, page_indices, ps, s, positions) -> np.ndarray:
    """Flat rows ``page*ps + offset`` of sequence-local key positions."""
    cu, pi, pos = _i64(cu_kv_lens), _i64(page_indices), _i64(positions).reshape(-1)
    out = np.empty(len(pos), np.int64)
    _load().orc_physical_rows(_p(cu), _p(pi), int(ps), int(s), _p(pos), len(pos), _p(out))
    return out


# ---------------------------------------------------------------- a7
class ShareMapError(ValueError):
    pass


def build_index_share_map(indexer_types, skip_offset, num_layers):
    """ref.py, build_index_share_map: returns (full_slot {layer: slot},
    src_slot {layer: slot}, number of full layers)."""
    del skip_offset
    codes = {"full": 0, "shared": 1}
    types = None if indexer_types is None else np.array([codes.get(k, 2) for k in indexer_types], np.int32)
    full = np.empty(max(1, num_layers), np.int64)
    src = np.empty(max(1, num_layers), np.int64)
    nfull = np.zeros(1, np.int64)
    rc = _load().orc_share_map(None if types is None else _p(types), 0 if types is None else len(types),
                               int(num_layers), _p(full), _p(src), _p(nfull))
    if rc == 1:
        raise ShareMapError("indexer_types length != num_layers")
    if rc == 2:
        raise ShareMapError("a shared layer has no preceding full layer")
    if rc == 3:
        raise ShareMapError("unknown indexer type")
    full_slot = {l: int(full[l]) for l in range(num_layers) if full[l] >= 0}
    src_slot = {l: int(src[l]) for l in range(num_layers)}
    return full_slot, src_slot, int(nfull[0])


# ---------------------------------------------------------------- a1 - a3
def indexer_score_row(q_t, w_t, keys) -> np.ndarray:
    """Scores of one query ([H, D], weights [H]) against ``keys`` [n, D]."""
    q, qd = _typed(q_t)
    w, wd = _typed(w_t)
    k, kd = _typed(keys)
    H, D = q.shape
    n = k.shape[0]
    out = np.empty(n, np.float32)
    _load().orc_score_row(_p(q), qd, _p(w), wd, _p(k), kd, H, D, n, _p(out))
    return out


def _score_matrix(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens):
    toks = _tokens(tokens, cu_q_lens)
    meta = _meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    kc, kd = _typed(kcache)
    P, ps, D = kc.shape
    if len(toks) == 0:
        return np.zeros((0, 1), np.float32), np.zeros(0, np.int64), toks, ps
    qr, qd = _typed(_rows(q, toks))
    wr, wd = _typed(_rows(w, toks))
    H = qr.shape[1]
    nvis = _geometry(meta[0], meta[1])[2][toks]
    ld = max(1, int(nvis.max()))
    out = np.full((len(toks), ld), np.nan, np.float32)
    lens = np.empty(len(toks), np.int64)
    _load().orc_indexer_scores(_p(qr), qd, _p(wr), wd, _p(kc), kd, ps, H, D, *map(_p, meta), len(meta[1]) - 1,
                               _p(toks), len(toks), ld, _p(out), _p(lens))
    return out, lens, toks, ps


def indexer_scores(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens=None):
    """Score rows for the given tokens (all by default): row ``t`` holds the
    scores of its visible prefix; masked positions are absent."""
    out, lens, _, _ = _score_matrix(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens)
    return [out[i, : lens[i]] for i in range(len(lens))]


def topk_of_row(scores, k) -> np.ndarray:
    """Exact top-k of one row (finite entries by (score desc, index asc),
    ``min(k, n)`` of them, ascending, -1 padded)."""
    s = _f32(scores)
    out = np.empty((1, k), np.int64)
    _load().orc_topk_rows(_p(s), max(1, len(s)), _p(_i64([len(s)])), 1, k, _p(out))
    return out[0].astype(np.int32)


def page_scores_of_row(scores, ps) -> np.ndarray:
    """Max-pool of one score row per page of ``ps`` positions."""
    s = _f32(scores)
    out = np.empty(-(-len(s) // ps), np.float32)
    _load().orc_page_scores_row(_p(s), len(s), int(ps), _p(out))
    return out


def page_topk_of_row(scores, ps, k_pages) -> np.ndarray:
    """Top ``k_pages`` pages of one row by max-pooled score."""
    s = _f32(scores)
    out = np.empty((1, k_pages), np.int64)
    _load().orc_page_topk_rows(_p(s), max(1, len(s)), _p(_i64([len(s)])), 1, int(ps), k_pages, _p(out))
    return out[0].astype(np.int32)


def topk_rows_of(rows, k) -> np.ndarray:
    """Exact top-k [n, k] int32 of a list of score rows (as topk_of_row)."""
    n = len(rows)
    lens = _i64([len(r) for r in rows])
    ld = max(1, int(lens.max()) if n else 1)
    mat = np.zeros((n, ld), np.float32)
    for i, r in enumerate(rows):
        mat[i, : len(r)] = r
    out = np.empty((n, k), np.int64)
    if n:
        _load().orc_topk_rows(_p(mat), ld, _p(lens), n, k, _p(out))
    return out.astype(np.int32)


def indexer_topk(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, k, tokens=None):
    """(token top-k [n, k] int32, score rows) of the given tokens."""
    out, lens, toks, _ = _score_matrix(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens)
    sel = np.empty((len(toks), k), np.int64)
    if len(toks):
        _load().orc_topk_rows(_p(out), out.shape[1], _p(lens), len(toks), k, _p(sel))
    return sel.astype(np.int32), [out[i, : lens[i]] for i in range(len(lens))]


def indexer_page_topk(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, k_pages, tokens=None):
    """(page top-k [n, k_pages] int32, score rows) of the given tokens."""
    out, lens, toks, ps = _score_matrix(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, tokens)
    sel = np.empty((len(toks), k_pages), np.int64)
    if len(toks):
        _load().orc_page_topk_rows(_p(out), out.shape[1], _p(lens), len(toks), ps, k_pages, _p(sel))
    return sel.astype(np.int32), [out[i, : lens[i]] for i in range(len(lens))]


# ---------------------------------------------------------------- a4
def lift_units(topk_units, cu_q_lens, cu_kv_lens, ps) -> np.ndarray:
    """Sequence-local page ids -> global page-table keys (-1 stays -1)."""
    tk = _i64(topk_units)
    cu_q = _i64(cu_q_lens)
    out = np.empty(tk.shape, np.int64)
    _load().orc_lift_units(_p(tk), tk.shape[0], tk.shape[1], _p(cu_q), len(cu_q) - 1, _p(_i64(cu_kv_lens)),
                           int(ps), _p(out))
    return out


def block_union(units_global, QB, u_max):
    """build_block_unit_tables: (units [nQB, u_max] int32, member
    [nQB, QB, u_max] int8, counts [nQB] int32)."""
    g = _i64(units_global)
    T, K = g.shape
    nqb = -(-T // QB) if T else 0
    units = np.empty((nqb, u_max), np.int32)
    member = np.empty((nqb, QB, u_max), np.int8)
    counts = np.empty(nqb, np.int32)
    if nqb:
        _load().orc_block_union(_p(g), T, K, QB, u_max, _p(units), _p(member), _p(counts))
    return units, member, counts


# ---------------------------------------------------------------- a5 / a6
def selected_positions(sel_row, unit, ps) -> np.ndarray:
    """Key positions named by one selection row (tokens, or whole pages)."""
    del ps
    sel = _i64(sel_row).reshape(-1)
    out = np.empty(max(1, len(sel) * unit), np.int64)
    n = _load().orc_selected_positions(_p(sel), len(sel), int(unit), _p(out))
    return out[:n]


def _attend_inputs(q, kv, toks):
    qr, qd = _typed(_rows(q, toks))
    kvc, kvd = _typed(kv)
    P, ps, W = kvc.shape
    return qr, qd, kvc, kvd, ps, W


def sparse_mla(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, sel, unit, sm_scale, Dv, tokens=None):
    """sparse_mla_ref over the selections: fp64 ``o [n, H, Dv]``, ``lse [n, H]``."""
    toks = _tokens(tokens, cu_q_lens)
    meta = _meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    qr, qd, kvc, kvd, ps, W = _attend_inputs(q, kv, toks)
    H, Dk = qr.shape[1], qr.shape[2]
    sr = _i64(_rows(sel, toks)).reshape(len(toks), -1)
    o = np.empty((len(toks), H, Dv), np.float64)
    lse = np.empty((len(toks), H), np.float64)
    if len(toks):
        _load().orc_sparse_mla(_p(qr), qd, _p(kvc), kvd, ps, W, H, Dk, Dv, *map(_p, meta), len(meta[1]) - 1,
                               _p(toks), len(toks), _p(sr), sr.shape[1], int(unit), float(sm_scale), _p(o), _p(lse))
    return o, lse


def qblock_attend(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, units, member, counts, QB, sm_scale, Dv,
                  tokens=None):
    """_qblock_kernel semantics over the block unions: fp64 ``o``, ``lse``."""
    toks = _tokens(tokens, cu_q_lens)
    meta = _meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    qr, qd, kvc, kvd, ps, W = _attend_inputs(q, kv, toks)
    H, Dk = qr.shape[1], qr.shape[2]
    un = _i64(units)
    mem = np.ascontiguousarray(np.asarray(member, dtype=np.int8))
    cnt = _i64(counts)
    o = np.empty((len(toks), H, Dv), np.float64)
    lse = np.empty((len(toks), H), np.float64)
    if len(toks):
        _load().orc_qblock_attend(_p(qr), qd, _p(kvc), kvd, ps, W, H, Dk, Dv, *map(_p, meta), len(meta[1]) - 1,
                                  _p(toks), len(toks), _p(un), _p(mem), _p(cnt), int(QB), un.shape[1],
                                  float(sm_scale), _p(o), _p(lse))
    return o, lse


def dense_mla(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, sm_scale, Dv, tokens=None,
              sliding_window=None, soft_cap=None):
    """Dense causal MLA (optional sliding window and tanh logit cap): fp64 ``o``."""
    toks = _tokens(tokens, cu_q_lens)
    meta = _meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    qr, qd, kvc, kvd, ps, W = _attend_inputs(q, kv, toks)
    H, Dk = qr.shape[1], qr.shape[2]
    o = np.empty((len(toks), H, Dv), np.float64)
    if len(toks):
        _load().orc_dense_mla(_p(qr), qd, _p(kvc), kvd, ps, W, H, Dk, Dv, *map(_p, meta), len(meta[1]) - 1,
                              _p(toks), len(toks), float(sm_scale), int(sliding_window or 0), float(soft_cap or 0.0),
                              _p(o))
    return o


# ------------------------------------------ the step before the path, and next rows
def paged_write_back(cache, rows, seq_lens, cu_q_lens, cu_kv_lens, page_indices):
    """Copy of ``cache`` [P, ps, W] with every query token's row written into
    its own slot (_scatter_paged); the input is not modified."""
    out = np.array(cache, copy=True, order="C")
    src = np.ascontiguousarray(np.asarray(rows).astype(out.dtype))
    P, ps, W = out.shape
    D = src.shape[1]
    meta = _meta(seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T = int(meta[1][-1])
    if T:
        _load().orc_paged_write_back(_p(out), out.itemsize, ps, W, _p(src), D, *map(_p, meta), len(meta[1]) - 1, T)
    return out


def topk_pages_of_tokens(topk_row, ps, cap):
    """(ascending unique pages of one query's tokens, first ``cap``, -1
    padded; the uncapped number of pages)."""
    row = _i64(topk_row).reshape(-1)
    out = np.empty(cap, np.int64)
    n = _load().orc_topk_pages_of_tokens(_p(row), len(row), int(ps), int(cap), _p(out))
    return out, int(n)


def approx_topk_of_row(scores, k, over):
    """Two-stage approximate top-k of one row (strided bins of
    ``min(n, over*k)``, exact top-k of the bin maxima), ascending, -1 padded."""
    s = _f32(scores)
    out = np.empty(k, np.int64)
    _load().orc_approx_topk_row(_p(s), len(s), int(k), int(over), _p(out))
    return out

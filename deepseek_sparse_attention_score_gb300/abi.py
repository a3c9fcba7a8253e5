"""Thin Python binding of the C ABI in ``include/dsa.h``.

Every function here has the name of the C entry point it wraps and does
argument marshalling only: shape/dtype/device checks, optional allocation of
output and workspace tensors with PyTorch, the ctypes call on the current CUDA
stream, and turning a negative return code into an exception. All arithmetic
runs in the CUDA kernels of ``libdsa_gb300.so``; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa_gb300.so")

ERRORS = {
    -1: "DSA_ERR_INVALID_ARGUMENT",
    -2: "DSA_ERR_UNSUPPORTED",
    -3: "DSA_ERR_WORKSPACE",
    -4: "DSA_ERR_CUDA",
    -5: "DSA_ERR_SHARED_BEFORE_FULL",
    -6: "DSA_ERR_BAD_INDEXER_TYPE",
    -7: "DSA_ERR_ALIGNMENT",
    -8: "DSA_ERR_SCRATCH_LIMIT",
}
STATUS_UNION_TRUNCATED = 0x1
STATUS_BAD_METADATA = 0x2
STATUS_BAD_INDEX = 0x4
STATUS_TIMEOUT = 0x8
STATUS_INTERNAL = 0x10

EXPORTS = (
    "dsa_index_build_share_map",
    "dsa_indexer_workspace_size",
    "dsa_indexer_topk",
    "dsa_indexer_page_topk",
    "dsa_build_block_union",
    "dsa_sparse_mla_decode_workspace_size",
    "dsa_sparse_mla_decode",
    "dsa_sparse_mla_prefill_qblock",
    "dsa_sparse_mla_prefill_qblock_range",
    "dsa_paged_write_back",
    "dsa_paged_write_back_pair",
    "dsa_dense_mla",
    "dsa_selftest_wait_timeout",
    "dsa_indexer_topk_approx_workspace_size",
    "dsa_indexer_topk_approx",
    "dsa_topk_pages_from_tokens",
    "dsa_device_sm_count",
    "dsa_launch_count",
    "dsa_sparse_mla_decode_noalloc",
)


class DSAError(RuntimeError):
    def __init__(self, fn, rc):
        super().__init__(f"{fn} returned {rc} ({ERRORS.get(rc, 'unknown')})")
        self.rc = rc


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_F = ctypes.c_float


def lib() -> ctypes.CDLL:
    """Load the in-tree library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(there is no non-CUDA implementation of this package)")
    L = ctypes.CDLL(LIB_PATH)
    L.dsa_index_build_share_map.argtypes = [_P, _I, _I, _P, _P, _P]
    L.dsa_indexer_workspace_size.argtypes = [_I, _I, _I, _I]
    L.dsa_indexer_workspace_size.restype = _Z
    L.dsa_indexer_topk.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P,
                                   _Z, _P]
    L.dsa_indexer_page_topk.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I,
                                        _P, _P, _P, _Z, _P]
    L.dsa_build_block_union.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P]
    L.dsa_sparse_mla_decode_workspace_size.argtypes = [_I, _I, _I]
    L.dsa_sparse_mla_decode_workspace_size.restype = _Z
    L.dsa_sparse_mla_decode.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                        _F, _P, _P, _P, _Z, _P]
    L.dsa_sparse_mla_prefill_qblock.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                                _I, _I, _I, _I, _F, _P, _P, _P]
    L.dsa_sparse_mla_prefill_qblock_range.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                                      _I, _I, _I, _I, _I, _F, _I, _I, _P, _P, _P]
    L.dsa_sparse_mla_decode_noalloc.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                                _I, _I, _F, _P, _P, _P]
    L.dsa_paged_write_back.argtypes = [_P, _P, _I, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]
    L.dsa_paged_write_back_pair.argtypes = [_P, _P, _I, _I, _P, _I, _P, _I, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I,
                                            _I, _P]
    L.dsa_topk_pages_from_tokens.argtypes = [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P]
    L.dsa_dense_mla.argtypes = [_P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _F,
                                _P, _P, _P, _Z, _P]
    L.dsa_indexer_topk_approx_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I]
    L.dsa_indexer_topk_approx_workspace_size.restype = _Z
    L.dsa_indexer_topk_approx.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                          _P, _P, _Z, _P]
    L.dsa_selftest_wait_timeout.argtypes = [_P, ctypes.c_longlong, _P]
    L.dsa_device_sm_count.argtypes = []
    L.dsa_launch_count.argtypes = []
    L.dsa_launch_count.restype = ctypes.c_longlong
    for name in EXPORTS:
        if name not in ("dsa_indexer_workspace_size", "dsa_sparse_mla_decode_workspace_size",
                        "dsa_launch_count", "dsa_indexer_topk_approx_workspace_size"):
            getattr(L, name).restype = _I
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise DSAError(fn, rc)


def _need(t, name, dtype, device, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _meta(device, seq_lens, cu_q_lens, cu_kv_lens, page_indices):
    for n, t in (("seq_lens", seq_lens), ("cu_q_lens", cu_q_lens), ("cu_kv_lens", cu_kv_lens),
                 ("page_indices", page_indices)):
        _need(t, n, torch.int32, device, 1)
    return seq_lens.numel(), page_indices.numel()


# --------------------------------------------------------------------- host
def dsa_index_build_share_map(indexer_types, num_layers, skip_offset=0):
    """IndexShare layer -> slot map. ``indexer_types``: sequence of 0 (full) /
    1 (shared), or None for all full. Returns (full_slot, src_slot, num_full)
    as Python lists / int (full_slot is -1 on shared layers)."""
    L = lib()
    types = None
    if indexer_types is not None:
        types = (ctypes.c_int32 * num_layers)(*[int(x) for x in indexer_types])
    full = (ctypes.c_int32 * max(1, num_layers))()
    src = (ctypes.c_int32 * max(1, num_layers))()
    nf = ctypes.c_int32(0)
    rc = L.dsa_index_build_share_map(types, num_layers, skip_offset, full, src, ctypes.byref(nf))
    _check("dsa_index_build_share_map", rc)
    return list(full)[:num_layers], list(src)[:num_layers], nf.value


def dsa_indexer_workspace_size(T, S, max_kv, ps):
    return int(lib().dsa_indexer_workspace_size(T, S, max_kv, ps))


def dsa_sparse_mla_decode_workspace_size(T, H, Dv=512):
    return int(lib().dsa_sparse_mla_decode_workspace_size(T, H, Dv))


def dsa_device_sm_count():
    return int(lib().dsa_device_sm_count())


def dsa_launch_count():
    return int(lib().dsa_launch_count())


# ------------------------------------------------------------------ indexer
def dsa_indexer_topk(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, *, k, max_kv, topk=None,
                     topk_scores=None, want_scores=False, ws=None, dev_status=None):
    """Indexer score + exact token top-k. Returns ``topk`` (and the scores of
    the selected positions when ``want_scores`` or ``topk_scores`` is given)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(w, "w", torch.float32, dev, 2)
    _need(kcache, "kcache", torch.bfloat16, dev, 3)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, Hi, Di = q.shape
    P, ps, _ = kcache.shape
    if topk is None:
        topk = torch.empty((T, k), dtype=torch.int32, device=dev)
    if want_scores and topk_scores is None:
        topk_scores = torch.empty((T, k), dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(max(1, dsa_indexer_workspace_size(T, S, max_kv, ps)), dtype=torch.uint8, device=dev)
    rc = lib().dsa_indexer_topk(_stream(dev), _ptr(q), _ptr(w), _ptr(kcache), _ptr(seq_lens), _ptr(cu_q_lens),
                                _ptr(cu_kv_lens), _ptr(page_indices), T, S, P, PTW, ps, Hi, Di, max_kv, k,
                                _ptr(topk), _ptr(topk_scores), _ptr(ws), ws.numel(), _ptr(dev_status))
    _check("dsa_indexer_topk", rc)
    return (topk, topk_scores) if topk_scores is not None else topk


def dsa_indexer_page_topk(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, *, k_pages, max_kv,
                          topk_pages=None, k=0, topk=None, with_tokens=False, topk_scores=None, ws=None,
                          dev_status=None):
    """Indexer score + page top-k (max-pooled per page); with ``with_tokens``
    (or a ``topk`` tensor) also the token top-k from the same score pass.
    Returns ``topk_pages`` or ``(topk_pages, topk)``."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(w, "w", torch.float32, dev, 2)
    _need(kcache, "kcache", torch.bfloat16, dev, 3)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, Hi, Di = q.shape
    P, ps, _ = kcache.shape
    if topk_pages is None:
        topk_pages = torch.empty((T, k_pages), dtype=torch.int32, device=dev)
    if with_tokens and topk is None:
        topk = torch.empty((T, k), dtype=torch.int32, device=dev)
    if ws is None:
        ws = torch.empty(max(1, dsa_indexer_workspace_size(T, S, max_kv, ps)), dtype=torch.uint8, device=dev)
    rc = lib().dsa_indexer_page_topk(_stream(dev), _ptr(q), _ptr(w), _ptr(kcache), _ptr(seq_lens),
                                     _ptr(cu_q_lens), _ptr(cu_kv_lens), _ptr(page_indices), T, S, P, PTW, ps, Hi,
                                     Di, max_kv, k_pages, _ptr(topk_pages), k, _ptr(topk), _ptr(topk_scores),
                                     _ptr(ws), ws.numel(), _ptr(dev_status))
    _check("dsa_indexer_page_topk", rc)
    return (topk_pages, topk) if topk is not None else topk_pages


# -------------------------------------------------------------------- union
def dsa_build_block_union(topk_units, *, QB, u_max=0, cu_q_lens=None, cu_kv_lens=None, ps=64, PTW,
                          units=None, member=None, counts=None, dev_status=None):
    """Per-block sorted union, bit-packed slot-major membership and true
    counts. Returns (units [nQB,u_max], member [nQB,u_max,QB/32] int32 view of
    the uint32 words, counts [nQB])."""
    dev = topk_units.device
    _need(topk_units, "topk_units", torch.int32, dev, 2)
    T, K = topk_units.shape
    S = 0
    if cu_q_lens is not None:
        _need(cu_q_lens, "cu_q_lens", torch.int32, dev, 1)
        _need(cu_kv_lens, "cu_kv_lens", torch.int32, dev, 1)
        S = cu_q_lens.numel() - 1
    if u_max <= 0:
        u_max = min(QB * K, PTW)
    nqb = (T + QB - 1) // QB
    if units is None:
        units = torch.empty((nqb, u_max), dtype=torch.int32, device=dev)
    if member is None:
        member = torch.empty((nqb, u_max, QB // 32), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty((nqb,), dtype=torch.int32, device=dev)
    rc = lib().dsa_build_block_union(_stream(dev), _ptr(topk_units), T, K, QB, u_max, _ptr(cu_q_lens),
                                     _ptr(cu_kv_lens), S, ps, PTW, _ptr(units), _ptr(member), _ptr(counts),
                                     _ptr(dev_status))
    _check("dsa_build_block_union", rc)
    return units, member, counts


# ------------------------------------------------------------------- attend
def dsa_sparse_mla_decode(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, sel, *, unit, sm_scale, o=None,
                          lse=None, want_lse=False, ws=None, dev_status=None, Dv=512):
    """Sparse absorbed-MLA attention over per-query selections (token ids when
    ``unit == 1``, sequence-local pages when ``unit == page_size``)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(kv, "kv", torch.bfloat16, dev, 3)
    _need(sel, "sel", torch.int32, dev, 2)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, H, Dk = q.shape
    P, ps, row_stride = kv.shape
    K = sel.shape[1]
    if o is None:
        o = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
    if want_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if ws is None:
        nb = dsa_sparse_mla_decode_workspace_size(T, H, Dv)
        ws = torch.empty(max(1, nb), dtype=torch.uint8, device=dev)
    rc = lib().dsa_sparse_mla_decode(_stream(dev), _ptr(q), _ptr(kv), row_stride, _ptr(seq_lens), _ptr(cu_q_lens),
                                     _ptr(cu_kv_lens), _ptr(page_indices), _ptr(sel), K, unit, T, S, P, PTW, ps, H,
                                     Dk, Dv, float(sm_scale), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                     _ptr(dev_status))
    _check("dsa_sparse_mla_decode", rc)
    return (o, lse) if lse is not None else o


def dsa_sparse_mla_prefill_qblock(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, units, member, counts, *,
                                  QB, sm_scale, o=None, lse=None, want_lse=False, dev_status=None, Dv=512,
                                  t_range=None):
    """Query-block sparse-MLA prefill over the union tables of
    ``dsa_build_block_union`` (same QB and u_max). ``t_range=(b, e)``
    computes only the output rows of tokens b .. e-1
    (``dsa_sparse_mla_prefill_qblock_range``)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(kv, "kv", torch.bfloat16, dev, 3)
    _need(units, "units", torch.int32, dev, 2)
    _need(member, "member", torch.int32, dev, 3)
    _need(counts, "counts", torch.int32, dev, 1)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, H, Dk = q.shape
    P, ps, row_stride = kv.shape
    u_max = units.shape[1]
    if o is None:
        o = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
    if want_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if t_range is None:
        rc = lib().dsa_sparse_mla_prefill_qblock(_stream(dev), _ptr(q), _ptr(kv), row_stride, _ptr(seq_lens),
                                                 _ptr(cu_q_lens), _ptr(cu_kv_lens), _ptr(page_indices), _ptr(units),
                                                 _ptr(member), _ptr(counts), QB, u_max, T, S, P, PTW, ps, H, Dk, Dv,
                                                 float(sm_scale), _ptr(o), _ptr(lse), _ptr(dev_status))
        _check("dsa_sparse_mla_prefill_qblock", rc)
    else:
        rc = lib().dsa_sparse_mla_prefill_qblock_range(
            _stream(dev), _ptr(q), _ptr(kv), row_stride, _ptr(seq_lens), _ptr(cu_q_lens), _ptr(cu_kv_lens),
            _ptr(page_indices), _ptr(units), _ptr(member), _ptr(counts), QB, u_max, T, S, P, PTW, ps, H, Dk, Dv,
            float(sm_scale), int(t_range[0]), int(t_range[1]), _ptr(o), _ptr(lse), _ptr(dev_status))
        _check("dsa_sparse_mla_prefill_qblock_range", rc)
    return (o, lse) if lse is not None else o


def dsa_sparse_mla_decode_noalloc(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, sel, *, unit, sm_scale,
                                  o=None, lse=None, want_lse=False, dev_status=None, Dv=512):
    """Same result as :func:`dsa_sparse_mla_decode`, without a workspace.

    For callers that cannot allocate device memory on this path, for example a
    plugin that is handed only its input and output buffers. The library keeps
    its split scratch in a built-in 24 MiB device array. The first call on a
    device looks up that array's address (make it before any stream capture),
    calls that overlap on the GPU race on the array, and a problem needing more
    scratch raises DSA_ERR_SCRATCH_LIMIT. ``o``/``lse`` may be preallocated by
    the caller; when omitted they are allocated here with PyTorch (the library
    call itself allocates nothing)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(kv, "kv", torch.bfloat16, dev, 3)
    _need(sel, "sel", torch.int32, dev, 2)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, H, Dk = q.shape
    P, ps, row_stride = kv.shape
    K = sel.shape[1]
    if o is None:
        o = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
    if want_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    rc = lib().dsa_sparse_mla_decode_noalloc(_stream(dev), _ptr(q), _ptr(kv), row_stride, _ptr(seq_lens),
                                             _ptr(cu_q_lens), _ptr(cu_kv_lens), _ptr(page_indices), _ptr(sel), K,
                                             unit, T, S, P, PTW, ps, H, Dk, Dv, float(sm_scale), _ptr(o), _ptr(lse),
                                             _ptr(dev_status))
    _check("dsa_sparse_mla_decode_noalloc", rc)
    return (o, lse) if lse is not None else o


# ------------------------------------------------------------ write-back
def dsa_paged_write_back(rows, cache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, *, D=None, dev_status=None):
    """Write each query token's row (``rows`` [T, W], its first ``D`` columns)
    into its slot of the paged ``cache`` [P, ps, W'] in place."""
    dev = cache.device
    _need(rows, "rows", torch.bfloat16, dev, 2)
    _need(cache, "cache", torch.bfloat16, dev, 3)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, src_stride = rows.shape
    P, ps, cache_stride = cache.shape
    if D is None:
        D = min(src_stride, cache_stride)
    rc = lib().dsa_paged_write_back(_stream(dev), _ptr(rows), src_stride, D, _ptr(cache), cache_stride,
                                    _ptr(seq_lens), _ptr(cu_q_lens), _ptr(cu_kv_lens), _ptr(page_indices), T, S, P,
                                    PTW, ps, _ptr(dev_status))
    _check("dsa_paged_write_back", rc)
    return cache


def dsa_paged_write_back_pair(rows0, cache0, rows1, cache1, seq_lens, cu_q_lens, cu_kv_lens, page_indices, *,
                              D0=None, D1=None, dev_status=None):
    """Both caches (sharing one page table) in one launch: the first ``D0``
    columns of ``rows0`` into ``cache0`` and the first ``D1`` of ``rows1``
    into ``cache1``, in place."""
    dev = cache0.device
    _need(rows0, "rows0", torch.bfloat16, dev, 2)
    _need(cache0, "cache0", torch.bfloat16, dev, 3)
    _need(rows1, "rows1", torch.bfloat16, dev, 2)
    _need(cache1, "cache1", torch.bfloat16, dev, 3)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, s0 = rows0.shape
    T1, s1 = rows1.shape
    P, ps, c0 = cache0.shape
    P1, ps1, c1 = cache1.shape
    if T1 != T or P1 != P or ps1 != ps:
        raise ValueError("dsa_paged_write_back_pair: both targets need the same tokens, pages and page size")
    D0 = min(s0, c0) if D0 is None else D0
    D1 = min(s1, c1) if D1 is None else D1
    rc = lib().dsa_paged_write_back_pair(_stream(dev), _ptr(rows0), s0, D0, _ptr(cache0), c0, _ptr(rows1), s1, D1,
                                         _ptr(cache1), c1, _ptr(seq_lens), _ptr(cu_q_lens), _ptr(cu_kv_lens),
                                         _ptr(page_indices), T, S, P, PTW, ps, _ptr(dev_status))
    _check("dsa_paged_write_back_pair", rc)
    return cache0, cache1


def dsa_topk_pages_from_tokens(topk, *, ps, max_pages, cap=512, pages=None, counts=None, dev_status=None):
    """Ascending unique pages of each query's selected tokens, the first
    ``cap`` of them, -1 padded; returns ``(pages [T, cap], counts [T])`` with
    the uncapped number of unique pages per row."""
    dev = topk.device
    _need(topk, "topk", torch.int32, dev, 2)
    T, K = topk.shape
    if pages is None:
        pages = torch.empty((T, cap), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty((T,), dtype=torch.int32, device=dev)
    rc = lib().dsa_topk_pages_from_tokens(_stream(dev), _ptr(topk), T, K, ps, max_pages, cap, _ptr(pages),
                                          _ptr(counts), _ptr(dev_status))
    _check("dsa_topk_pages_from_tokens", rc)
    return pages, counts


def dsa_dense_mla(q, kv, seq_lens, cu_q_lens, cu_kv_lens, page_indices, *, max_kv, sm_scale, sliding_window=0,
                  soft_cap=0.0, o=None, lse=None, want_lse=False, ws=None, dev_status=None, Dv=512):
    """Dense causal absorbed-MLA over every visible position (optionally the
    ``sliding_window`` most recent ones, with a tanh logit cap)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(kv, "kv", torch.bfloat16, dev, 3)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, H, Dk = q.shape
    P, ps, row_stride = kv.shape
    if o is None:
        o = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
    if want_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if ws is None:
        nb = dsa_sparse_mla_decode_workspace_size(T, H, Dv)
        ws = torch.empty(max(1, nb), dtype=torch.uint8, device=dev)
    rc = lib().dsa_dense_mla(_stream(dev), _ptr(q), _ptr(kv), row_stride, _ptr(seq_lens), _ptr(cu_q_lens),
                             _ptr(cu_kv_lens), _ptr(page_indices), int(max_kv), T, S, P, PTW, ps, H, Dk, Dv,
                             float(sm_scale), int(sliding_window), float(soft_cap), _ptr(o), _ptr(lse), _ptr(ws),
                             ws.numel(), _ptr(dev_status))
    _check("dsa_dense_mla", rc)
    return (o, lse) if lse is not None else o


def dsa_indexer_topk_approx(q, w, kcache, seq_lens, cu_q_lens, cu_kv_lens, page_indices, *, k, max_kv, over=4,
                            topk=None, ws=None, dev_status=None):
    """Approximate token top-k: exact top-k of per-bin maxima over
    ``min(n, over * k)`` strided bins of each score row (ascending
    positions, -1 padded)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(w, "w", torch.float32, dev, 2)
    _need(kcache, "kcache", torch.bfloat16, dev, 3)
    S, PTW = _meta(dev, seq_lens, cu_q_lens, cu_kv_lens, page_indices)
    T, Hi, Di = q.shape
    P, ps, _ = kcache.shape
    if topk is None:
        topk = torch.empty((T, k), dtype=torch.int32, device=dev)
    if ws is None:
        nb = lib().dsa_indexer_topk_approx_workspace_size(T, S, max_kv, ps, k, over)
        ws = torch.empty(max(1, nb), dtype=torch.uint8, device=dev)
    rc = lib().dsa_indexer_topk_approx(_stream(dev), _ptr(q), _ptr(w), _ptr(kcache), _ptr(seq_lens), _ptr(cu_q_lens),
                                       _ptr(cu_kv_lens), _ptr(page_indices), T, S, P, PTW, ps, Hi, Di, int(max_kv),
                                       int(k), int(over), _ptr(topk), _ptr(ws), ws.numel(), _ptr(dev_status))
    _check("dsa_indexer_topk_approx", rc)
    return topk


def dsa_selftest_wait_timeout(dev_status, limit_clocks=2_000_000):
    """Run one bounded wait that is bound to run out (a barrier nothing
    arrives on); the device status word gets DSA_STATUS_TIMEOUT."""
    _need(dev_status, "dev_status", torch.int32, dev_status.device, 1)
    rc = lib().dsa_selftest_wait_timeout(_stream(dev_status.device), int(limit_clocks), _ptr(dev_status))
    _check("dsa_selftest_wait_timeout", rc)

"""Host-side checks that need no GPU: the library loads, exports every
symbol include/dsa.h declares, and the host-only entry points behave."""
import re
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_score_gb300 as m

    return m


def test_library_exports_every_declared_symbol(dsa):
    with open(os.path.join(ROOT, "include", "dsa.h")) as f:
        header = f.read()
    declared = set(re.findall(r"DSA_API\s+[\w ]+?\b(dsa_\w+)\(", header))
    assert len(declared) >= 9
    L = dsa.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert declared == set(dsa.abi.EXPORTS) | (declared - set(dsa.abi.EXPORTS))
    assert set(dsa.abi.EXPORTS) <= declared


def test_share_map_matches_closed_form(dsa):
    full, src, n = dsa.dsa_index_build_share_map([0, 1, 1, 0], 4)
    assert full == [0, -1, -1, 1] and src == [0, 0, 0, 1] and n == 2
    full, src, n = dsa.dsa_index_build_share_map(None, 3, skip_offset=7)
    assert full == [0, 1, 2] and src == [0, 1, 2] and n == 3


@pytest.mark.parametrize("types,code", [([1, 0], -5), ([0, 2], -6)])
def test_share_map_errors(dsa, types, code):
    with pytest.raises(dsa.DSAError) as e:
        dsa.dsa_index_build_share_map(types, len(types))
    assert e.value.rc == code


def test_share_map_agrees_with_oracle(dsa):
    import itertools
    import oracle as O

    names = {0: "full", 1: "shared"}
    for L in range(1, 6):
        for types in itertools.product([0, 1], repeat=L):
            try:
                ofull, osrc, on = O.build_index_share_map([names[t] for t in types], 0, L)
            except O.ShareMapError:
                with pytest.raises(dsa.DSAError):
                    dsa.dsa_index_build_share_map(list(types), L)
                continue
            full, src, n = dsa.dsa_index_build_share_map(list(types), L)
            assert n == on and src == [osrc[i] for i in range(L)]
            assert full == [ofull.get(i, -1) for i in range(L)]


def test_workspace_sizes_are_host_computable(dsa):
    a = dsa.dsa_indexer_workspace_size(32, 32, 8192, 64)
    b = dsa.dsa_indexer_workspace_size(64, 32, 8192, 64)
    assert 0 < a < b
    assert dsa.dsa_indexer_workspace_size(32, 32, 8192, 48) == 0  # unsupported page size


def test_selftest_wait_timeout_validates_on_host(dsa):
    import ctypes

    L = dsa.lib()
    fake = ctypes.c_void_p(16)  # never dereferenced: the arguments are rejected first
    assert L.dsa_selftest_wait_timeout(None, 0, fake) == -1
    assert L.dsa_selftest_wait_timeout(None, 10**11, fake) == -1
    assert L.dsa_selftest_wait_timeout(None, 1000, None) == -1


# ---------------------------------------------------------------- host checks
# Every case below is rejected (or, for T == 0, accepted as a no-op) before
# the library makes any CUDA call, so the fake device pointers are never
# dereferenced and no GPU is needed. The codes are the ones include/dsa.h
# documents.
OK, INVALID, UNSUPPORTED, WORKSPACE, ALIGNMENT = 0, -1, -2, -3, -7


def _ptr(addr=4096):
    import ctypes

    return ctypes.c_void_p(addr)


def _decode_args(**kw):
    a = dict(stream=None, q=_ptr(), kv=_ptr(), row_stride=576, seq_lens=_ptr(), cu_q_lens=_ptr(),
             cu_kv_lens=_ptr(), page_indices=_ptr(), sel=_ptr(), K=64, unit=1, T=4, S=4, P=16, PTW=16, ps=64,
             H=128, Dk=576, Dv=512, sm_scale=0.1, o=_ptr(), lse=None, ws=_ptr(), ws_bytes=1 << 20,
             dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(ps=48), UNSUPPORTED),               # page sizes 32, 64, 128 only
    (dict(row_stride=600), UNSUPPORTED),      # latent rows of 576 or 640
    (dict(Dv=256), UNSUPPORTED),
    (dict(Dk=512), UNSUPPORTED),
    (dict(unit=7), INVALID),                  # unit is 1 (tokens) or ps (pages)
    (dict(K=0), INVALID),
    (dict(sel=None), INVALID),
    (dict(sm_scale=float("nan")), INVALID),
    (dict(q=_ptr(4098)), ALIGNMENT),
    (dict(o=None), INVALID),
    (dict(seq_lens=None), INVALID),
    (dict(T=-1), INVALID),
    (dict(T=0, S=0, P=0, PTW=0), OK),         # nothing to do, nothing enqueued
])
def test_sparse_mla_decode_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_sparse_mla_decode(*_decode_args(**kw)) == code


def _dense_args(**kw):
    a = dict(stream=None, q=_ptr(), kv=_ptr(), row_stride=576, seq_lens=_ptr(), cu_q_lens=_ptr(),
             cu_kv_lens=_ptr(), page_indices=_ptr(), max_kv=1024, T=4, S=4, P=16, PTW=16, ps=64, H=128, Dk=576,
             Dv=512, sm_scale=0.1, sliding_window=0, soft_cap=0.0, o=_ptr(), lse=None, ws=_ptr(),
             ws_bytes=1 << 20, dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(sliding_window=-1), INVALID),
    (dict(soft_cap=-1.0), INVALID),
    (dict(soft_cap=float("inf")), INVALID),
    (dict(max_kv=0), INVALID),
    (dict(ps=100), UNSUPPORTED),
    (dict(kv=_ptr(4100)), ALIGNMENT),
    (dict(T=0, S=0, P=0, PTW=0), OK),
])
def test_dense_mla_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_dense_mla(*_dense_args(**kw)) == code


def _write_back_args(**kw):
    a = dict(stream=None, rows=_ptr(), src_stride=576, D=576, cache=_ptr(), cache_stride=576, seq_lens=_ptr(),
             cu_q_lens=_ptr(), cu_kv_lens=_ptr(), page_indices=_ptr(), T=4, S=4, P=16, PTW=16, ps=64,
             dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(D=100), UNSUPPORTED),               # rows move in 16-byte pieces
    (dict(D=640, src_stride=576), UNSUPPORTED),
    (dict(cache_stride=580), UNSUPPORTED),
    (dict(rows=None), INVALID),
    (dict(page_indices=None), INVALID),
    (dict(ps=0), INVALID),
    (dict(cache=_ptr(4104)), ALIGNMENT),
    (dict(T=-2), INVALID),
    (dict(T=0), OK),
    (dict(D=0), OK),
])
def test_paged_write_back_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_paged_write_back(*_write_back_args(**kw)) == code


def _write_back_pair_args(**kw):
    a = dict(stream=None, rows0=_ptr(), src_stride0=576, D0=576, cache0=_ptr(), cache_stride0=576, rows1=_ptr(),
             src_stride1=128, D1=128, cache1=_ptr(), cache_stride1=128, seq_lens=_ptr(), cu_q_lens=_ptr(),
             cu_kv_lens=_ptr(), page_indices=_ptr(), T=4, S=4, P=16, PTW=16, ps=64, dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(D1=100), UNSUPPORTED),              # each target moves in 16-byte pieces
    (dict(D0=640, src_stride0=576), UNSUPPORTED),
    (dict(cache_stride1=132), UNSUPPORTED),
    (dict(rows1=None), INVALID),              # a second cache without its rows
    (dict(cache0=None), INVALID),
    (dict(page_indices=None), INVALID),
    (dict(cache1=_ptr(4104)), ALIGNMENT),
    (dict(T=-1), INVALID),
    (dict(T=0), OK),
    (dict(D0=0, D1=0), OK),
])
def test_paged_write_back_pair_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_paged_write_back_pair(*_write_back_pair_args(**kw)) == code


def _pages_args(**kw):
    a = dict(stream=None, topk=_ptr(), T=4, K=64, ps=64, max_pages=1024, cap=512, pages=_ptr(), counts=None,
             dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(cap=0), INVALID),
    (dict(ps=0), INVALID),
    (dict(K=-1), INVALID),
    (dict(max_pages=0), UNSUPPORTED),
    (dict(max_pages=(1 << 20) + 1), UNSUPPORTED),
    (dict(pages=None), INVALID),
    (dict(topk=None), INVALID),
    (dict(T=0), OK),
])
def test_topk_pages_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_topk_pages_from_tokens(*_pages_args(**kw)) == code


def _approx_args(**kw):
    a = dict(stream=None, q=_ptr(), w=_ptr(), kcache=_ptr(), seq_lens=_ptr(), cu_q_lens=_ptr(), cu_kv_lens=_ptr(),
             page_indices=_ptr(), T=4, S=4, P=16, PTW=16, ps=64, Hi=32, Di=128, max_kv=1024, k=64, over=4,
             topk=_ptr(), ws=_ptr(), ws_bytes=1 << 30, dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(over=0), INVALID),
    (dict(k=0), INVALID),
    (dict(topk=None), INVALID),
    (dict(Hi=16), UNSUPPORTED),               # 32 indexer heads of 128 dims
    (dict(Di=64), UNSUPPORTED),
    (dict(k=16385), UNSUPPORTED),             # the sort of the winners holds 16 K
    (dict(ws=None), WORKSPACE),
    (dict(ws_bytes=16), WORKSPACE),
    (dict(w=_ptr(4108)), ALIGNMENT),
    (dict(T=0, S=0, P=0, PTW=0), OK),
])
def test_indexer_topk_approx_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_indexer_topk_approx(*_approx_args(**kw)) == code


def _indexer_args(**kw):
    a = dict(stream=None, q=_ptr(), w=_ptr(), kcache=_ptr(), seq_lens=_ptr(), cu_q_lens=_ptr(), cu_kv_lens=_ptr(),
             page_indices=_ptr(), T=4, S=4, P=16, PTW=16, ps=64, Hi=32, Di=128, max_kv=1024, k=64, topk=_ptr(),
             topk_scores=None, ws=_ptr(), ws_bytes=1 << 30, dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(topk=None), INVALID),
    (dict(k=0), INVALID),
    (dict(max_kv=0), INVALID),
    (dict(Hi=64), UNSUPPORTED),
    (dict(ps=16), UNSUPPORTED),
    (dict(ws=None), WORKSPACE),
    (dict(ws_bytes=64), WORKSPACE),
    (dict(kcache=_ptr(4112 + 4)), ALIGNMENT),
    (dict(cu_kv_lens=None), INVALID),
    (dict(T=0, S=0, P=0, PTW=0), OK),
])
def test_indexer_topk_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_indexer_topk(*_indexer_args(**kw)) == code


def _union_args(**kw):
    a = dict(stream=None, topk_units=_ptr(), T=64, K=4, QB=32, u_max=0, cu_q_lens=_ptr(), cu_kv_lens=_ptr(), S=2,
             ps=64, PTW=16, units=_ptr(), member=_ptr(), counts=_ptr(), dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(QB=48), INVALID),                   # query blocks of a multiple of 32 tokens
    (dict(QB=2048), INVALID),
    (dict(K=0), INVALID),
    (dict(PTW=0), INVALID),
    (dict(cu_kv_lens=None), INVALID),
    (dict(member=None), INVALID),
    (dict(T=0), OK),
])
def test_block_union_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_build_block_union(*_union_args(**kw)) == code


def _qblock_args(**kw):
    a = dict(stream=None, q=_ptr(), kv=_ptr(), row_stride=576, seq_lens=_ptr(), cu_q_lens=_ptr(),
             cu_kv_lens=_ptr(), page_indices=_ptr(), units=_ptr(), member=_ptr(), counts=_ptr(), QB=32, u_max=64,
             T=64, S=2, P=16, PTW=16, ps=64, H=128, Dk=576, Dv=512, sm_scale=0.1, o=_ptr(), lse=None,
             dev_status=None)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,code", [
    (dict(QB=40), INVALID),
    (dict(u_max=0), INVALID),
    (dict(counts=None), INVALID),
    (dict(sm_scale=float("inf")), INVALID),
    (dict(row_stride=512), UNSUPPORTED),
    (dict(o=_ptr(4120 + 2)), ALIGNMENT),
    (dict(T=0, S=0, P=0, PTW=0), OK),
])
def test_prefill_qblock_host_checks(dsa, kw, code):
    assert dsa.lib().dsa_sparse_mla_prefill_qblock(*_qblock_args(**kw)) == code


def _qblock_range_args(t_begin, t_end, **kw):
    a = _qblock_args(**kw)
    # the range goes between sm_scale and o
    return a[:22] + [t_begin, t_end] + a[22:]


@pytest.mark.parametrize("tb,te,code", [
    (-1, 8, INVALID),
    (8, 4, INVALID),
    (0, 65, INVALID),
    (5, 5, OK),      # an empty range enqueues nothing
])
def test_prefill_qblock_range_host_checks(dsa, tb, te, code):
    assert dsa.lib().dsa_sparse_mla_prefill_qblock_range(*_qblock_range_args(tb, te)) == code
